"""Numerical stress cases of the decode kernels against the oracle.

The read path (news article "超越 TurboQuant…", section "OSCAR 的设计思路":
unpack, restore scale/zero, floating-point accumulation) feeds the tensor cores
fp16 operands: key codes as fp16 subnormals against hi/lo query fragments,
value codes against p * scale rounded to fp16, and, in the shared-prefix
kernel, weights that are rescaled lazily (only when the running maximum grows
by more than 2^8). These cases move the logits far from the default scale:

* peaked: sm_scale x 8, a few tokens carry nearly all of the weight;
* diffuse: sm_scale / 8, the weights are almost uniform;
* aligned: one query head is a multiple of a history key with the outlier
  channels, so a single token takes almost all of the weight;
* equal: the query is zero, every logit is 0 and the output is the plain mean.

Every case runs on the CUDA-core decoder, the per-request mma.sync and tcgen05
decoders and the shared-prefix tensor-core decoder (followed by either
per-request decoder), on fp32 output, against the oracle's
fp64 attention over the pool bytes the GPU wrote, with the decode tolerance
(per (request, q-head) row, max |o - ref| / max |ref| <= 2e-3).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import bit_kv_cache_decode_gb300 as osc
    from gpu_cases import build_decode_case, pool_from_device, queries, row_rel_err, to_dev_bf16, tokens
import synth
from oracle import attention as A

TOL = 2e-3
SHARED = 64 + 64 * 24                     # shared prefix: the sink page and 24 history pages
LENS = [SHARED + 64 * 6 + 37 + 256, SHARED + 64 * 2 + 256, SHARED + 300]
KERNELS = [pytest.param((0, 0), id="simt"), pytest.param((1, 0), id="mma"), pytest.param((1, 24), id="shared"),
           pytest.param((2, 0), id="tc"), pytest.param((2, 24), id="shared_tc")]
CASES = ["peaked", "diffuse", "aligned", "equal"]


def _queries(case, seed, hkv, gq):
    q = queries(seed, 0, hkv, gq, batch=len(LENS))
    sm = synth.sm_scale()
    if case == "peaked":
        sm *= 8.0
    elif case == "diffuse":
        sm /= 8.0
    elif case == "aligned":
        # head 0 of each kv head of request 0: 4 x a history key (position 64 + 130, in the shared prefix);
        # head 1 of request 1: 2 x a key of its own history
        k0, _ = tokens(seed, 0, hkv, SHARED, extra=0)
        k1, _ = tokens(seed, 0, hkv, LENS[1], extra=2)
        for h in range(hkv):
            q[0, h * gq] = synth.bf16_round(4.0 * k0[64 + 130, h])
            q[1, h * gq + 1] = synth.bf16_round(2.0 * k1[SHARED + 70, h])
    elif case == "equal":
        q[0] = 0.0
    return q, sm


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("case", CASES)
def test_decode_stress(kernel, case):
    algo, shared_pages = kernel
    hkv, gq, seed, v_mode = 2, 4, 31, 0
    cache, prm, hp, bp = build_decode_case(LENS, hkv, gq, v_mode, seed, shared_prefix=SHARED, algo=algo)
    q, sm = _queries(case, seed, hkv, gq)
    out = cache.decode_attention(0, to_dev_bf16(q), np.array(LENS, np.int32), hp, bp, sm, out_dtype=osc.OUT_FP32,
                                 shared_hist_pages=shared_pages)
    assert cache.get_status() == 0
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    pm = pool_from_device(cache, 0)
    for r, L in enumerate(LENS):
        ref, _ = A.decode_request(q[r], L, pm, hp[r], bp[r], prm, True, sm)
        err = row_rel_err(got[r], ref)
        assert err.max() <= TOL, (case, r, err.max())
