"""Parity at the bench's full sizes and in its launch configuration: the workloads
bench.py times, built by its own workload builder, stepped with the same
oscar_decode_step calls per layer (same kernels, split policy and kernel builds;
the bench replays them from a CUDA graph), then sampled outputs checked against
the oracle's fp64 attention over the pool bytes the GPU wrote.

* Qwen3-8B full stack: 36 layers x (32 q / 8 kv heads), batch 1, 102,400-token
  context; layers 0, 17 and 35 checked after two steps.
* the same stack in explicit-V mode (raw V in the cache, rotated back in the
  merge); layers 0 and 35 checked after two steps.
* Qwen3-4B batched: 36 layers, batch 32 x 102,400 tokens sharing a 92,160-token
  prefix (the shared-prefix kernel for the shared pages); layers 0 and 35,
  requests 0, 13 and 31 checked after two steps.

Tolerance as everywhere: bf16 outputs within one bf16 ulp of the reference plus
2e-3 of the row's largest magnitude."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import bench
    import bit_kv_cache_decode_gb300 as osc
    from gpu_cases import DEV, bf16_ulp, pool_from_device
import synth
from oracle import attention as A
from oracle import pool as P

TOL = 2e-3


def _run_steps(wl, steps: int, seed: int):
    """`steps` decode steps of every layer exactly as the bench issues them; returns the last step's
    queries [layers, B, Hq, 128] (bf16 values as float64) and outputs, and the final lengths."""
    cache, nl, B, H, hq = wl["cache"], wl["layers"], wl["B"], wl["H"], wl["hq"]
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    seq = torch.from_numpy(wl["lens"].astype(np.int32)).to(DEV)
    out = torch.empty(nl, B, hq, 128, dtype=torch.bfloat16, device=DEV)
    for _ in range(steps):
        kv = torch.randn(nl, 2, B, H, 128, generator=g, device=DEV).to(torch.bfloat16)
        q = torch.randn(nl, B, hq, 128, generator=g, device=DEV).to(torch.bfloat16)
        for layer in range(nl):
            cache.decode_step(layer, q[layer], kv[layer, 0], kv[layer, 1], seq, wl["hist_pt"], wl["bf16_pt"],
                              synth.sm_scale(), out=out[layer], shared_hist_pages=wl["shp"])
        seq.add_(1)
    torch.cuda.synchronize()
    assert cache.get_status() == 0
    return q.double().cpu().numpy(), out.double().cpu().numpy(), seq.cpu().numpy()


def _check(wl, qn, on, lens, layers, requests):
    H = wl["H"]
    for layer in layers:
        pm = pool_from_device(wl["cache"], layer)
        cs = wl["cals"][layer * H:(layer + 1) * H]
        prm = [P.HeadParams(c["U_K"], c["U_V"], c["tau_K"], c["tau_V"]) for c in cs]
        for r in requests:
            ref, _ = A.decode_request(qn[layer, r], int(lens[r]), pm, wl["hist_np"][r], wl["bf16_np"][r], prm,
                                      wl["cfg"].v_mode == osc.V_ABSORBED, synth.sm_scale())
            got = on[layer, r]
            slack = TOL * np.abs(ref).max(axis=-1, keepdims=True)
            bad = np.abs(got - ref) > bf16_ulp(ref) + slack
            assert not bad.any(), (layer, r, float((np.abs(got - ref) / np.abs(ref).max(-1, keepdims=True)).max()))


def test_qwen3_8b_36_layers_100k_context():
    wl = bench.build_workload("qwen3_8b_36l", 1234, DEV, with_bf16=False, steps_capacity=8, algo=1)
    qn, on, lens = _run_steps(wl, 2, 77)
    _check(wl, qn, on, lens, layers=(0, 17, 35), requests=(0,))


def test_qwen3_8b_36_layers_100k_context_explicit_v():
    wl = bench.build_workload("qwen3_8b_36l", 1235, DEV, with_bf16=False, steps_capacity=8, algo=1, v_explicit=True)
    assert wl["cfg"].v_mode == osc.V_EXPLICIT
    qn, on, lens = _run_steps(wl, 2, 79)
    _check(wl, qn, on, lens, layers=(0, 35), requests=(0,))


def test_qwen3_4b_batch32_shared_prefix_100k_context():
    wl = bench.build_workload("qwen3_4b_b32", 1234, DEV, with_bf16=False, steps_capacity=8, algo=1)
    assert wl["shp"] > 0
    qn, on, lens = _run_steps(wl, 2, 78)
    _check(wl, qn, on, lens, layers=(0, 35), requests=(0, 13, 31))
