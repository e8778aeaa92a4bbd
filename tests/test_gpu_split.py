"""GPU parity of the fused pair kernel's split last round, through the C ABI.

When the last round of a launch's tiles would leave at least half of the
CTA pairs idle and K spans at least 128 K-blocks (32 with eight epilogue
warps), each of its tiles is computed as two halves of its K-blocks on two
pairs; the second half's fp32
accumulator reaches the tile's owner through global memory.  These cases make that happen on purpose (every tile split, a
tail of tiles split after whole rounds, an odd number of K-blocks, ragged H,
microchunks, FP8 operands) and hold the result to the same bar as every other
path.  Also: a row block with more N-tiles than the grid has pairs takes the
PIPELINED path instead of the fused kernel.
"""
import numpy as np
import pytest

import oracle
from synth import Workload, make_inputs, make_inputs_fp8

from .gpu_util import Run, plan
from .parity import compare

pytestmark = pytest.mark.gpu

fln = pytest.importorskip("decoder_layer_projection_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fln.build()
    fln.load()
    yield


_REF = {}


def _check(rb, ob, d, wl, name):
    if wl.name not in _REF:   # the oracle once per workload (K = 8192 takes a few seconds)
        _REF[wl.name] = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], wl.eps, wl.norm_kind)[:2]
    r, o = _REF[wl.name]
    compare(rb, r, name + " residual")
    compare(ob, o, name + " out")


WL = Workload("split", T=520, K=8192, H=512, eps=1e-5, r_sigma=2.0, seed=31)


# (tile, CTA target): 520 tokens = 3 row blocks of 256 (the last ragged); K = 8192 is 128 K-blocks;
# the split decision per launch
#   tile 128 / all SMs: 12 tiles, all split (24 pairs)
#   tile 128 / 16 CTAs: 8 pairs, one whole round of 8 tiles, the last 4 split
#   tile 128 / 20 CTAs: 10 pairs, 10 whole tiles, the last 2 split (2 whole tiles of their row block before)
#   tiles 256 / 224 / 192: 6 / 9 / 9 tiles, all split (224 and 192 leave a ragged last N-tile)
@pytest.mark.parametrize("tile,ctas", [(128, 0), (128, 16), (128, 20), (256, 0), (224, 0), (192, 0)])
def test_split_tiles_full_parity(tile, ctas):
    d = make_inputs(WL)
    run = Run(d, WL.eps, WL.norm_kind)
    rb, ob = run(plan(fln.PATH_FUSED, chunk=700, tile_n=tile, gemm_ctas=ctas))
    _check(rb, ob, d, WL, f"split tile={tile} ctas={ctas}")
    # deterministic: the owner adds the other half in a fixed order
    rb2, ob2 = run(plan(fln.PATH_FUSED, chunk=700, tile_n=tile, gemm_ctas=ctas))
    assert np.array_equal(rb, rb2) and np.array_equal(ob, ob2)


def test_split_changes_only_the_rounding():
    """14 CTAs (7 pairs): 12 tiles leave 5 for the last round, too many to split; 16 CTAs split 4.
    Both meet the oracle's bar; they differ in some bits, since the split tiles add two fp32 halves (if
    they were identical everywhere, the split would not have run)."""
    d = make_inputs(WL)
    run = Run(d, WL.eps, WL.norm_kind)
    whole = run(plan(fln.PATH_FUSED, chunk=700, tile_n=128, gemm_ctas=14))
    split = run(plan(fln.PATH_FUSED, chunk=700, tile_n=128, gemm_ctas=16))
    _check(*whole, d, WL, "unsplit")
    _check(*split, d, WL, "split")
    assert not np.array_equal(whole[0], split[0])


def test_split_odd_k_blocks_ragged_h_gemma():
    # K = 8256: 129 K-blocks, halves of 64 and 65; H = 264: the second N-tile is 8 columns wide
    wl = Workload("split_odd", T=300, K=8256, H=264, norm_kind=1, eps=1e-6, gamma_mode="plain", seed=32)
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    for tile in (256, 128):
        rb, ob = run(plan(fln.PATH_FUSED, chunk=300, tile_n=tile))
        _check(rb, ob, d, wl, f"split odd K tile={tile}")


def test_split_with_small_microchunks():
    # chunks of 256, 256 and 8 tokens run back to back in one launch of 520 tokens, whose tiles all split
    d = make_inputs(WL)
    run = Run(d, WL.eps, WL.norm_kind)
    rb, ob = run(plan(fln.PATH_FUSED, chunk=256, tile_n=128))
    _check(rb, ob, d, WL, "split chunks of 256")


# Eight epilogue warps (two groups on alternate tiles): a helper's half goes out before it takes the
# output staging, so the split runs from 32 K-blocks and with no guard on the round before.
WL8 = Workload("split_two_groups", T=520, K=2048, H=512, eps=1e-5, r_sigma=2.0, seed=36)
WL8_GUARD = Workload("split_two_groups_guard", T=700, K=2048, H=2048, norm_kind=1, eps=1e-6, gamma_mode="plain",
                     seed=37)


# (workload, tile, CTA target): WL8 has 3 x 2 tiles (256) or 3 x 3 (224): all split on the full grid; on 8
# CTAs (4 pairs) 4 whole tiles then 2 split.  WL8_GUARD: 3 x 8 tiles on 10 pairs, 20 whole then 4 split,
# with 4 whole tiles of the split row block in the round before (the one-group kernel would not split).
@pytest.mark.parametrize("wl,tile,ctas", [(WL8, 256, 0), (WL8, 224, 0), (WL8, 256, 8), (WL8_GUARD, 256, 20)],
                         ids=["256-all", "224-all", "256-tail", "guard"])
def test_two_group_split_full_parity(wl, tile, ctas):
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    rb, ob = run(plan(fln.PATH_FUSED, chunk=1024, tile_n=tile, gemm_ctas=ctas, epi_warps=8))
    _check(rb, ob, d, wl, f"two-group split tile={tile} ctas={ctas}")
    rb2, ob2 = run(plan(fln.PATH_FUSED, chunk=1024, tile_n=tile, gemm_ctas=ctas, epi_warps=8))
    assert np.array_equal(rb, rb2) and np.array_equal(ob, ob2)
    # four epilogue warps do not split at 32 K-blocks: the same bar, other rounding on the split tiles
    w4 = run(plan(fln.PATH_FUSED, chunk=1024, tile_n=tile, gemm_ctas=ctas, epi_warps=4))
    _check(*w4, d, wl, f"one group tile={tile} ctas={ctas}")
    assert not np.array_equal(rb, w4[0])


def test_two_group_split_with_microchunks_and_repeats():
    # chunks of 128 tokens grouped in one launch; repeated calls agree bit for bit (generation-tagged halves)
    d = make_inputs(WL8)
    run = Run(d, WL8.eps, WL8.norm_kind)
    res = [run(plan(fln.PATH_FUSED, chunk=c, tile_n=256, epi_warps=8)) for c in (128, 520, 128)]
    for rb, ob in res[1:]:
        assert np.array_equal(rb, res[0][0]) and np.array_equal(ob, res[0][1])
    _check(*res[0], d, WL8, "two-group split, chunks of 128")


WL_LONG = Workload("split_long", T=16388, K=8192, H=256, eps=1e-5, r_sigma=2.0, seed=35)


def test_split_in_every_launch_of_a_long_call():
    """16388 tokens: a launch of 16384 (64 row-pair blocks x 2 N-tiles on 64 pairs, no split) and a tail
    launch of 4 tokens (2 tiles, split), for chunks of 4096, 1024 and 256 alike (whole chunks are grouped
    up to 16384 tokens a launch).  Every row against the oracle; the chunkings agree bit for bit; rows
    past the call stay unwritten (Run's guard rows)."""
    d = make_inputs(WL_LONG)
    run = Run(d, WL_LONG.eps, WL_LONG.norm_kind)
    res = [run(plan(fln.PATH_FUSED, chunk=c, tile_n=128, gemm_ctas=128)) for c in (4096, 1024, 256)]
    for rb, ob in res[1:]:
        assert np.array_equal(rb, res[0][0]) and np.array_equal(ob, res[0][1])
    rows = np.arange(WL_LONG.T)
    r, o, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], WL_LONG.eps, WL_LONG.norm_kind,
                                      rows=rows)
    compare(res[0][0][rows], r, "two launches residual")
    compare(res[0][1][rows], o, "two launches out")


@pytest.mark.parametrize("tile,ew", [(128, 4), (256, 8)])
def test_split_fp8(tile, ew):
    torch = pytest.importorskip("torch")
    from .gpu_util import dev_bf16, host_bits
    # E4M3 K-blocks hold 128 elements: K = 16384 is 128 of them
    wl = Workload("split_fp8", T=300, K=16384, H=640, eps=1e-5, r_sigma=2.0, seed=33)
    d = make_inputs_fp8(wl)
    K, H = wl.K, wl.H
    x = torch.from_numpy(np.ascontiguousarray(d["x8"])).cuda()
    W = torch.from_numpy(np.ascontiguousarray(d["W8"])).cuda()
    sx = torch.from_numpy(np.ascontiguousarray(d["x_scale"])).cuda()
    sw = torch.from_numpy(np.ascontiguousarray(d["w_scale"])).cuda()
    gamma = torch.from_numpy(np.ascontiguousarray(d["gamma"], np.float32)).cuda()
    # one epilogue group from 128 K-blocks, two groups from 32: both split every tile here
    fln.fln_set_plan(K, H, wl.norm_kind, plan(fln.PATH_FUSED, chunk=300, tile_n=tile, epi_warps=ew),
                     dtype=fln.DTYPE_E4M3)
    try:
        r = dev_bf16(d["r0"])
        out = torch.empty_like(r)
        fln.fused_proj_add_rmsnorm_fp8(x, sx, W, sw, r, gamma, wl.eps, wl.norm_kind, 0, out)
        fln.fln_device_status()
    finally:
        fln.fln_set_plan(K, H, wl.norm_kind, None, dtype=fln.DTYPE_E4M3)
    ro, oo, _ = oracle.proj_add_rmsnorm_fp8(d["x8"], d["x_scale"], d["W8"], d["w_scale"], d["r0"], d["gamma"],
                                            wl.eps, wl.norm_kind)
    compare(host_bits(r), ro, f"split fp8 tile={tile} ew={ew} residual")
    compare(host_bits(out), oo, f"split fp8 tile={tile} ew={ew} out")


@pytest.mark.parametrize("tile", [128, 224])
def test_row_block_wider_than_the_grid_takes_the_pipelined_path(tile):
    # H = 2048 in 16 (tile 128) or 10 (tile 224) N-tiles on 4 pairs: the fused kernel would need every
    # N-tile of a row block on its own pair, so the call runs GEMM -> slot -> add + norm instead
    wl = Workload("wide_rows", T=300, K=256, H=2048, eps=1e-5, r_sigma=2.0, seed=34)
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    fln.fln_profile_enable(True)
    try:
        rb, ob = run(plan(fln.PATH_FUSED, chunk=300, tile_n=tile, gemm_ctas=8))
        prof = fln.fln_profile_read()
    finally:
        fln.fln_profile_enable(False)
    _check(rb, ob, d, wl, f"wide rows tile={tile}")
    assert prof["gemm_fused"]["launches"] == 0
    assert prof["gemm_slot"]["launches"] == 1 and prof["norm_slot"]["launches"] == 1
