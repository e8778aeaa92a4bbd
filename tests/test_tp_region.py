"""The TPSP region's host logic on CPU (no GPU): the token partition, padding,
rank offsets and chunk order that fused_proj_rs_add_rmsnorm_ag follows, taken
from the library's own host functions.

* Partition invariants over a grid of (T, P, microchunk): every token is
  owned by exactly one (rank, chunk), shards are contiguous and padded to
  ceil(T / P) rows, block rows agree across ranks, chunks run in order.
* Two gloo ranks run the whole region as the library schedules it -- each
  rank's K-shard partial projection of every rank's rows of a chunk, a
  reduce-scatter over tokens, the add + norm of its valid rows, an all-gather
  and the scatter back to token order -- with the arithmetic in float64, and
  the result is compared with the fp64 oracle of the undivided region.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import decoder_layer_projection_gb300 as fln
import oracle
from synth import Workload, bf16_bits_to_f32, make_inputs


def _owners(T, P, c):
    S, cs, nch = fln.fln_tp_layout(T, P, c)
    seen = np.zeros(T, np.int64)
    for q in range(P):
        last = -1
        for i in range(nch):
            tok0, n, valid = fln.fln_tp_chunk_rows(T, P, c, i, q)
            assert n == fln.fln_tp_chunk_rows(T, P, c, i, 0)[1]  # same block rows on every rank
            assert 0 <= valid <= n <= cs
            if valid:
                assert tok0 == q * S + i * cs            # rank offset + chunk offset
                assert tok0 > last                       # chunks in token order
                last = tok0 + valid - 1
                assert q * S <= tok0 and tok0 + valid <= min((q + 1) * S, T)
                seen[tok0:tok0 + valid] += 1
        assert sum(fln.fln_tp_chunk_rows(T, P, c, i, q)[1] for i in range(nch)) == S  # padded shard
    return seen, S, cs, nch


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
def test_partition_covers_every_token_once(P):
    fln.build()
    for T in (1, 2, 7, 8, 37, 100, 129, 1000, 4097, 10000):
        for c in (0, 1, 8, 100, 128, 4096):
            seen, S, cs, nch = _owners(T, P, c)
            assert np.all(seen == 1), (T, P, c)
            assert S == -(-T // P)
            assert cs == min(c or 1024, S)
            assert nch == -(-S // cs)


def test_partition_arguments():
    fln.build()
    assert fln.fln_tp_layout(0, 4, 0) == (0, 1, 0)
    for bad in ((5, 0, 0), (5, 2, -1), (5, 2, 4097), (-1, 2, 0)):
        with pytest.raises(fln.FlnError) as e:
            fln.fln_tp_layout(*bad)
        assert e.value.status == fln.FLN_ERR_INVALID_ARG
    with pytest.raises(fln.FlnError):
        fln.fln_tp_chunk_rows(37, 2, 8, 3, 0)   # only chunks 0..2
    with pytest.raises(fln.FlnError):
        fln.fln_tp_chunk_rows(37, 2, 8, 0, 2)   # only ranks 0..1


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


def _region_rank(rank, world, port, case, out):
    """One rank of the region, scheduled by the library's partition; float64 arithmetic."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl, chunk = case
        d = make_inputs(wl)
        T, K, H = wl.T, wl.K, wl.H
        Kp = K // world
        xp = _f64(d["x"])[:, rank * Kp:(rank + 1) * Kp]
        Wp = _f64(d["W"])[:, rank * Kp:(rank + 1) * Kp]
        g = d["gamma"].astype(np.float64) + (1.0 if wl.norm_kind else 0.0)
        S, cs, nch = fln.fln_tp_layout(T, world, chunk)
        # this rank's residual shard, padded to S rows
        shard = np.zeros((S, H))
        v0 = max(0, min(S, T - rank * S))
        shard[:v0] = _f64(d["r0"])[rank * S:rank * S + v0]
        outp = np.full((T, H), np.nan)
        for i in range(nch):
            # partial y of every rank's rows of the chunk (rank-major blocks; rows past T are zeros)
            blocks = []
            for q in range(world):
                tok0, n, _ = fln.fln_tp_chunk_rows(T, world, chunk, i, q)
                rows = np.zeros((n, Kp))
                first = q * S + i * cs
                m = max(0, min(n, T - first))
                rows[:m] = xp[first:first + m]
                blocks.append(rows @ Wp.T)
            slot = torch.from_numpy(np.stack(blocks))
            dist.all_reduce(slot)                      # reduce ...
            red = slot[rank].numpy()                   # ... scatter: this rank's block
            tok0, n, valid = fln.fln_tp_chunk_rows(T, world, chunk, i, rank)
            r = shard[i * cs:i * cs + valid] + red[:valid]
            shard[i * cs:i * cs + valid] = r
            send = np.zeros((n, H))
            send[:valid] = r / np.sqrt((r * r).mean(axis=1, keepdims=True) + wl.eps) * g
            gathered = [torch.zeros((n, H), dtype=torch.float64) for _ in range(world)]
            dist.all_gather(gathered, torch.from_numpy(send))
            for q in range(world):
                tq, _, vq = fln.fln_tp_chunk_rows(T, world, chunk, i, q)
                assert np.all(np.isnan(outp[tq:tq + vq]))   # each row written once
                outp[tq:tq + vq] = gathered[q][:vq].numpy()
        out[rank] = (shard[:v0].copy(), outp)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", [
    (Workload("tp_ragged", T=37, K=64, H=48, eps=1e-5, r_sigma=2.0, seed=51), 8),
    (Workload("tp_gemma", T=21, K=32, H=64, norm_kind=1, eps=1e-6, gamma_mode="plain", seed=52), 0),
    (Workload("tp_one_chunk_pad", T=5, K=16, H=24, eps=1e-5, seed=53), 4096),
], ids=lambda c: c[0].name if isinstance(c, tuple) else str(c))
def test_two_gloo_ranks_region_matches_the_oracle(case):
    fln.build()
    world = 2
    wl, _ = case
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_region_rank, args=(world, port, case, out), nprocs=world, join=True)
        res = dict(out)
    d = make_inputs(wl)
    r, o, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], wl.eps, wl.norm_kind)
    S = -(-wl.T // world)
    for rank in range(world):
        shard, outp = res[rank]
        assert not np.isnan(outp).any()                                   # every token gathered
        np.testing.assert_allclose(outp, o, rtol=1e-10, atol=1e-10)       # the undivided region
        np.testing.assert_allclose(shard, r[rank * S:rank * S + shard.shape[0]], rtol=1e-10, atol=1e-10)
