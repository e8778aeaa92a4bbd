"""GPU parity of the MoE region against the fp64 oracle, through the C ABI.

* routing: expert ids and the grouping (offsets, row_token, row_slot, row_of)
  bit for bit, gates within fp32 rounding, with planted equal logits;
* the grouped down projection + unpermute + add + norm on ragged shapes
  (K and H tails, experts without rows, one expert, k = 1..4), the same bar
  as the dense paths (tests/parity.py), guard rows after T untouched, on
  single CTAs and (256 or more rows per expert) on CTA pairs, with bad
  offsets caught on both;
* routing then the region chained on the device;
* the Mixtral-8x7B down shape at decode, 512 and 4096 tokens, every row;
* argument checks.
"""
import numpy as np
import pytest

import oracle
from synth import MOE_CONFIGS, Workload, make_inputs_moe

from .gpu_util import dev_bf16, host_bits
from .parity import compare

pytestmark = pytest.mark.gpu

fln = pytest.importorskip("decoder_layer_projection_gb300")
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fln.build()
    fln.load()
    yield


def _logits(T, E, seed):
    g = np.random.default_rng(seed)
    lg = g.standard_normal((T, E)).astype(np.float32)
    if T > 3:
        lg[1, :] = 0.5                      # every logit equal
        lg[2, E // 2] = lg[2, 0] = 7.0      # a tie for the top
        lg[3, ::2] = -1.25                  # ties lower down
    return lg


@pytest.mark.parametrize("T,E,k", [(1, 4, 1), (7, 8, 2), (300, 8, 2), (129, 64, 4), (1024, 256, 8), (33, 5, 5)])
def test_routing_matches_oracle(T, E, k):
    lg = _logits(T, E, seed=T + E + k)
    res = fln.fln_moe_route(torch.from_numpy(lg).cuda(), k)
    fln.fln_device_status()
    ids, w = oracle.moe_route(lg, k)
    np.testing.assert_array_equal(res["ids"].cpu().numpy(), ids)
    np.testing.assert_allclose(res["gates"].cpu().numpy(), w, rtol=2e-6, atol=1e-7)
    offsets, row_token, row_slot, row_of = oracle.moe_permute(ids, E)
    np.testing.assert_array_equal(res["offsets"].cpu().numpy(), offsets)
    np.testing.assert_array_equal(res["row_token"].cpu().numpy(), row_token)
    np.testing.assert_array_equal(res["row_slot"].cpu().numpy(), row_slot)
    np.testing.assert_array_equal(res["row_of"].cpu().numpy(), row_of)


class RunMoe:
    GUARD = 3

    def __init__(self, d, E, eps, kind):
        self.d, self.E, self.eps, self.kind = d, E, eps, kind
        self.T, self.k = d["ids"].shape
        self.offsets, _, _, self.row_of = oracle.moe_permute(d["ids"], E)
        self.hg = dev_bf16(d["hg"])
        self.We = torch.from_numpy(np.ascontiguousarray(d["We"]).view(np.int16)).view(torch.bfloat16).cuda()
        self.gamma = torch.from_numpy(np.ascontiguousarray(d["gamma"], np.float32)).cuda()

    def __call__(self):
        d = self.d
        H = d["We"].shape[1]
        r = dev_bf16(d["r0"], extra_rows=self.GUARD)
        out = dev_bf16(np.zeros((self.T, H), np.uint16), extra_rows=self.GUARD, fill_bits=0x7FC2)
        offs = torch.from_numpy(self.offsets).cuda()
        row_of = torch.from_numpy(self.row_of).cuda()
        gates = torch.from_numpy(d["wt"]).cuda()
        fln.fused_moe_down_add_rmsnorm(self.hg, offs, row_of, gates, self.We, r[:self.T], self.gamma, self.eps,
                                       self.kind, out=out[:self.T])
        fln.fln_device_status()
        rb, ob = host_bits(r), host_bits(out)
        assert np.all(rb[self.T:] == 0x7FC1), "residual guard rows were written"
        assert np.all(ob[self.T:] == 0x7FC2), "output guard rows were written"
        return rb[:self.T], ob[:self.T]

    def check(self, rb, ob, name, rows=None):
        d = self.d
        r, o, _ = oracle.moe_down_region(d["hg"], self.offsets, self.row_of, d["wt"], d["We"], d["r0"], d["gamma"],
                                         self.eps, self.kind)
        if rows is not None:
            r, o, rb, ob = r[rows], o[rows], rb[rows], ob[rows]
        compare(rb, r, name + " residual")
        compare(ob, o, name + " out")


SMALL = [
    (Workload("moe_a", T=24, K=256, H=256, eps=1e-6, r_sigma=1.0, seed=1), 4, 2),
    (Workload("moe_ragged", T=61, K=200, H=264, eps=1e-5, r_sigma=2.0, seed=2), 6, 3),
    (Workload("moe_one", T=5, K=136, H=520, eps=1e-5, r_sigma=2.0, seed=3), 1, 1),
    (Workload("moe_gemma", T=200, K=384, H=1032, norm_kind=1, eps=1e-6, gamma_mode="plain", seed=4), 8, 4),
    (Workload("moe_long_k", T=9, K=4104, H=512, eps=1e-5, r_sigma=2.0, seed=5), 8, 2),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: c[0].name)
def test_down_region_parity(case):
    wl, E, k = case
    d = make_inputs_moe(wl, E, k)
    run = RunMoe(d, E, wl.eps, wl.norm_kind)
    rb, ob = run()
    run.check(rb, ob, wl.name)
    rb2, ob2 = run()
    assert np.array_equal(rb, rb2) and np.array_equal(ob, ob2)


# At least 256 grouped rows per expert on average: the grouped GEMM runs on CTA pairs (256-row blocks that
# stop at each expert's end, 256-wide W tiles split between the two CTAs)
PAIR = [
    (Workload("moe_pair_ragged", T=600, K=200, H=264, eps=1e-5, r_sigma=2.0, seed=7), 2, 1),
    (Workload("moe_pair_gemma", T=300, K=448, H=520, norm_kind=1, eps=1e-6, gamma_mode="plain", seed=8), 4, 4),
    (Workload("moe_pair_top3", T=700, K=136, H=384, eps=1e-5, r_sigma=2.0, seed=9), 8, 3),
]


@pytest.mark.parametrize("case", PAIR, ids=lambda c: c[0].name)
def test_down_region_parity_on_cta_pairs(case):
    wl, E, k = case
    assert wl.T * k >= 256 * E
    d = make_inputs_moe(wl, E, k)
    run = RunMoe(d, E, wl.eps, wl.norm_kind)
    rb, ob = run()
    run.check(rb, ob, wl.name)
    rb2, ob2 = run()
    assert np.array_equal(rb, rb2) and np.array_equal(ob, ob2)


def test_expert_without_rows_on_cta_pairs():
    wl = Workload("moe_pair_empty", T=1100, K=256, H=384, eps=1e-5, r_sigma=2.0, seed=10)
    d = dict(make_inputs_moe(wl, 4, 1))
    g = np.random.default_rng(10)
    d["ids"] = g.choice([0, 1, 3], size=(wl.T, 1)).astype(np.int32)
    run = RunMoe(d, 4, wl.eps, wl.norm_kind)
    assert run.offsets[2] == run.offsets[3] and wl.T >= 256 * 4
    rb, ob = run()
    run.check(rb, ob, "expert without rows, CTA pairs")


def test_bad_offsets_on_cta_pairs_write_nothing():
    wl, E, k = PAIR[0]
    d = make_inputs_moe(wl, E, k)
    run = RunMoe(d, E, wl.eps, wl.norm_kind)
    T, H = d["r0"].shape
    good = run.offsets
    for bad in (np.array([0, good[1], good[2] + 128], np.int32), np.array([0, good[2], good[1]], np.int32)):
        r = dev_bf16(d["r0"])
        out = dev_bf16(np.full((T, H), 0x7FC2, np.uint16))
        fln.fused_moe_down_add_rmsnorm(run.hg, torch.from_numpy(bad).cuda(), torch.from_numpy(run.row_of).cuda(),
                                       torch.from_numpy(d["wt"]).cuda(), run.We, r, run.gamma, wl.eps,
                                       wl.norm_kind, out=out)
        _expect_bad_index()
        assert np.array_equal(host_bits(r), d["r0"]) and np.all(host_bits(out) == 0x7FC2)
    rb, ob = run()
    run.check(rb, ob, "after bad offsets, CTA pairs")


def test_expert_without_rows():
    wl = Workload("moe_empty", T=40, K=256, H=384, eps=1e-5, r_sigma=2.0, seed=6)
    d = dict(make_inputs_moe(wl, 8, 2))
    g = np.random.default_rng(6)
    d["ids"] = np.stack([g.choice([0, 1, 2, 4, 5, 6, 7], 2, replace=False) for _ in range(wl.T)]).astype(np.int32)
    run = RunMoe(d, 8, wl.eps, wl.norm_kind)
    assert run.offsets[3] == run.offsets[4]
    rb, ob = run()
    run.check(rb, ob, "expert without rows")


def test_route_then_region_on_device():
    wl, E, k = MOE_CONFIGS["moe_tiny"]
    d = make_inputs_moe(wl, E, k)
    lg = torch.from_numpy(d["logits"]).cuda()
    res = fln.fln_moe_route(lg, k)
    ids, w = oracle.moe_route(d["logits"], k)
    offsets, _, _, row_of = oracle.moe_permute(ids, E)
    # the grouped activations follow the device grouping (identical to the oracle's, checked above)
    r = dev_bf16(d["r0"])
    out = torch.empty_like(r)
    We = torch.from_numpy(np.ascontiguousarray(d["We"]).view(np.int16)).view(torch.bfloat16).cuda()
    gamma = torch.from_numpy(d["gamma"]).cuda()
    fln.fused_moe_down_add_rmsnorm(dev_bf16(d["hg"]), res["offsets"], res["row_of"], res["gates"], We, r, gamma,
                                   wl.eps, wl.norm_kind, out=out)
    fln.fln_device_status()
    ro, oo, _ = oracle.moe_down_region(d["hg"], offsets, row_of, w.astype(np.float32), d["We"], d["r0"], d["gamma"],
                                       wl.eps, wl.norm_kind)
    compare(host_bits(r), ro, "chained residual")
    compare(host_bits(out), oo, "chained out")


@pytest.mark.parametrize("name,T", [("mixtral_8x7b_down_decode", 8), ("mixtral_8x7b_down", 512),
                                    ("mixtral_8x7b_down", 4096)])
def test_full_size_every_row(name, T):
    # every token of the Mixtral-8x7B down region against the oracle (4096 tokens: the bench workload)
    wl, E, k = MOE_CONFIGS[name]
    d = make_inputs_moe(wl, E, k, T=T)
    run = RunMoe(d, E, wl.eps, wl.norm_kind)
    rb, ob = run()
    run.check(rb, ob, f"{name} T={T}")


def test_rejects_bad_arguments():
    lib = fln.load()
    assert lib.fln_moe_route(None, 4, 300, 2, None, None, None, None, None, None, None) == fln.FLN_ERR_INVALID_ARG
    assert lib.fln_moe_route(None, 4, 8, 9, None, None, None, None, None, None, None) == fln.FLN_ERR_INVALID_ARG
    assert lib.fln_moe_route(None, 4, 4, 5, None, None, None, None, None, None, None) == fln.FLN_ERR_INVALID_ARG
    rc = lib.fused_moe_down_add_rmsnorm(None, None, None, None, None, None, None, 1e-5, 0, 4, 100, 256, 8, 2, None, None)
    assert rc == fln.FLN_ERR_INVALID_ARG and "K=" in fln.fln_last_error()
    rc = lib.fused_moe_down_add_rmsnorm(None, None, None, None, None, None, None, 1e-5, 0, 4, 128, 20000, 8, 2, None,
                                        None)
    assert rc == fln.FLN_ERR_UNSUPPORTED


@pytest.mark.parametrize("T,E,k,H", [(1, 4, 1, 8), (300, 8, 2, 264), (129, 64, 4, 4096), (33, 5, 5, 1032)])
def test_gather_matches_oracle(T, E, k, H):
    lg = _logits(T, E, seed=3 * T + H)
    res = fln.fln_moe_route(torch.from_numpy(lg).cuda(), k)
    x = np.random.default_rng(T + H).integers(0, 1 << 16, size=(T, H), dtype=np.uint16)
    xg = fln.fln_moe_gather(dev_bf16(x), res["row_token"], k)
    fln.fln_device_status()
    ids, _ = oracle.moe_route(lg, k)
    _, row_token, _, _ = oracle.moe_permute(ids, E)
    assert np.array_equal(host_bits(xg), oracle.moe_gather(x, row_token))


def test_gather_argument_checks():
    lib = fln.load()
    assert lib.fln_moe_gather(None, None, 4, 2, 12, None, None) == fln.FLN_ERR_INVALID_ARG
    assert lib.fln_moe_gather(None, None, 4, 9, 16, None, None) == fln.FLN_ERR_INVALID_ARG
    assert lib.fln_moe_gather(None, None, 0, 2, 16, None, None) == fln.FLN_OK
    buf = torch.zeros((24, 16), dtype=torch.bfloat16, device="cuda")
    tok = torch.zeros((16,), dtype=torch.int32, device="cuda")
    with pytest.raises(fln.FlnError, match="overlaps"):
        fln.fln_moe_gather(buf[:8], tok, 2, out=buf[4:20])   # xg [16, 16] starts inside x [8, 16]


def _expect_bad_index():
    with pytest.raises(fln.FlnError) as ei:
        fln.fln_device_status()
    assert ei.value.status == fln.FLN_ERR_INVALID_ARG and "index out of range" in ei.value.message


def test_bad_device_indices_are_reported_and_skipped():
    """Indices that live in device memory (row_token, offsets, row_of) are checked by the kernels: the rows
    they touch are left unwritten, the status call reports it, and the next call runs normally."""
    wl, E, k = MOE_CONFIGS["moe_tiny"]
    d = make_inputs_moe(wl, E, k)
    T, H = d["r0"].shape
    # gather: two bad token indices
    x = np.random.default_rng(1).integers(0, 1 << 15, size=(T, H), dtype=np.uint16)
    _, row_token, _, _ = oracle.moe_permute(d["ids"], E)
    bad_tok = row_token.copy()
    bad_tok[1], bad_tok[4] = T, -1
    xg = dev_bf16(np.full((T * k, H), 0x7FC3, np.uint16))
    fln.fln_moe_gather(dev_bf16(x), torch.from_numpy(bad_tok).cuda(), k, out=xg)
    _expect_bad_index()
    got, want = host_bits(xg), oracle.moe_gather(x, row_token)
    assert np.all(got[[1, 4]] == 0x7FC3)
    keep = np.setdiff1d(np.arange(T * k), [1, 4])
    assert np.array_equal(got[keep], want[keep])
    # region: offsets that do not end at T * k -> nothing written, residual and out untouched
    run = RunMoe(d, E, wl.eps, wl.norm_kind)
    good = run.offsets
    bad_end = good.copy()
    bad_end[E] += 128
    r = dev_bf16(d["r0"])
    out = dev_bf16(np.full((T, H), 0x7FC2, np.uint16))
    fln.fused_moe_down_add_rmsnorm(run.hg, torch.from_numpy(bad_end).cuda(), torch.from_numpy(run.row_of).cuda(),
                                   torch.from_numpy(d["wt"]).cuda(), run.We, r, run.gamma, wl.eps, wl.norm_kind,
                                   out=out)
    _expect_bad_index()
    assert np.array_equal(host_bits(r), d["r0"]) and np.all(host_bits(out) == 0x7FC2)
    fln.fln_device_status()         # the error word was cleared by the report
    # region: offsets out of order
    run.offsets = good.copy()
    run.offsets[1], run.offsets[2] = good[2], good[1]
    assert run.offsets[1] != run.offsets[2]
    with pytest.raises(fln.FlnError, match="index out of range"):
        run()
    # region: one bad row_of entry -> that token's rows untouched, the others exact
    run.offsets = good
    bad_row = run.row_of.copy()
    bad_row[3, k - 1] = T * k
    r = dev_bf16(d["r0"])
    out = dev_bf16(np.full((T, H), 0x7FC2, np.uint16))
    fln.fused_moe_down_add_rmsnorm(run.hg, torch.from_numpy(good).cuda(), torch.from_numpy(bad_row).cuda(),
                                   torch.from_numpy(d["wt"]).cuda(), run.We, r, run.gamma, wl.eps, wl.norm_kind,
                                   out=out)
    _expect_bad_index()
    rb, ob = host_bits(r), host_bits(out)
    assert np.array_equal(rb[3], d["r0"][3]) and np.all(ob[3] == 0x7FC2)
    rb_ok, ob_ok = run()
    others = np.setdiff1d(np.arange(T), [3])
    assert np.array_equal(rb[others], rb_ok[others]) and np.array_equal(ob[others], ob_ok[others])
    run.check(rb_ok, ob_ok, "after bad indices")


def test_moe_path_graph_replay_is_bitwise():
    """Routing, gather and the down region captured in one CUDA graph: every replay gives the eager result
    (nothing is read back on the host between the steps, so the whole path captures), and that result is the
    oracle's with the gathered rows standing in for the expert activations."""
    wl, E, k = MOE_CONFIGS["moe_tiny"]
    d = make_inputs_moe(wl, E, k)
    T, K = d["hg"].shape[0] // k, d["We"].shape[2]
    x_np = np.random.default_rng(11).integers(0, 1 << 15, size=(T, K), dtype=np.uint16) & 0xBF7F  # finite
    x, lg = dev_bf16(x_np), torch.from_numpy(d["logits"]).cuda()
    We = torch.from_numpy(np.ascontiguousarray(d["We"]).view(np.int16)).view(torch.bfloat16).cuda()
    gamma = torch.from_numpy(d["gamma"]).cuda()
    r0 = dev_bf16(d["r0"])
    r, out = r0.clone(), torch.empty_like(r0)

    def step():
        res = fln.fln_moe_route(lg, k)
        xg = fln.fln_moe_gather(x, res["row_token"], k)
        fln.fused_moe_down_add_rmsnorm(xg, res["offsets"], res["row_of"], res["gates"], We, r, gamma, wl.eps,
                                       wl.norm_kind, out=out)
        return res

    step()                                   # eager; sizes the workspace
    fln.fln_device_status()
    r_eager, o_eager = host_bits(r), host_bits(out)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    r.copy_(r0)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        step()
    for _ in range(3):
        r.copy_(r0)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        fln.fln_device_status()
        assert np.array_equal(host_bits(r), r_eager) and np.array_equal(host_bits(out), o_eager)
    ids, w = oracle.moe_route(d["logits"], k)
    offsets, row_token, _, row_of = oracle.moe_permute(ids, E)
    ro, oo, _ = oracle.moe_down_region(oracle.moe_gather(x_np, row_token), offsets, row_of, w.astype(np.float32),
                                       d["We"], d["r0"], d["gamma"], wl.eps, wl.norm_kind)
    compare(r_eager, ro, "graph path residual")
    compare(o_eager, oo, "graph path out")
