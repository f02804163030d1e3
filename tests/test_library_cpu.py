"""CPU checks of the C-ABI library: it loads, exports every symbol the header
declares, validates layouts on the host, and its host-side calibration agrees
with the oracle. No GPU compute is called here."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import synth
from oracle import rotation

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def osc():
    import __graft_entry__
    __graft_entry__.build()
    import bit_kv_cache_decode_gb300 as o
    return o


def _declared():
    hdr = open(os.path.join(ROOT, "include", "oscar.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"\b(oscar_[a-z0-9_]+)\s*\(", hdr)))


def test_every_declared_symbol_is_exported(osc):
    names = _declared()
    assert len(names) >= 17
    out = subprocess.run(["nm", "-D", "--defined-only", osc.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(oscar_[a-z0-9_]+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    assert set(osc.EXPORTS) == set(names)
    lib = osc.lib()
    for n in names:
        assert getattr(lib, n) is not None


def test_error_strings(osc):
    lib = osc.lib()
    assert lib.oscar_error_string(0) == b"ok"
    assert b"orthogonal" in lib.oscar_error_string(osc.ERR_NOT_ORTHOGONAL)


def _bytes(osc, **kw):
    cfg = osc.CacheConfig(**{**dict(num_layers=2, num_kv_heads=8, num_q_heads=32, num_int2_pages=10,
                                    num_bf16_pages=5, max_batch=2, max_splits=16), **kw})
    lay = cfg.layout()
    pb, wb = ctypes.c_size_t(), ctypes.c_size_t()
    rc = osc.lib().oscar_cache_bytes(ctypes.byref(lay), ctypes.byref(pb), ctypes.byref(wb))
    return rc, pb.value, wb.value


@pytest.mark.parametrize("meta,block", [(0, 5120), (1, 4608)])
def test_layout_sizes(osc, meta, block):
    rc, pb, wb = _bytes(osc, meta_format=meta)
    assert rc == 0
    # per layer: INT2 blocks, BF16 blocks, and U_K, U_V, U_V^T, tau_K, tau_V, R_K and R_V fragments,
    # the compact format's 32 grid constants and R_K and R_V as three bf16 parts (98,304 bytes each) per
    # kv head
    per_layer = (10 * 8 * block) + (5 * 8 * 32768) + 8 * ((5 * 128 * 128 + 2 * 128 + 32) * 4 + 2 * 98304)
    assert pb >= 2 * per_layer and pb < 2 * per_layer + 2 * 3 * 256
    parts = 2 * 32 * (16 + 5) * 132 * 4          # history splits + 5 BF16 chunks per (request, q head)
    assert wb >= parts


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=64), -2), (dict(group=32), -2), (dict(page_size=32), -2),
    (dict(num_q_heads=24), -2), (dict(num_q_heads=30), -1), (dict(sink=65), -1), (dict(recent=0), -1),
    (dict(max_batch=0), -1), (dict(v_mode=7), -1), (dict(num_layers=0), -1), (dict(meta_format=3), -1),
])
def test_layout_validation(osc, kw, code):
    rc, _, _ = _bytes(osc, **kw)
    assert rc == code


def test_null_arguments_rejected_without_a_device(osc):
    lib = osc.lib()
    assert lib.oscar_cache_create(None, None, None, None) == osc.ERR_INVALID_ARG
    assert lib.oscar_decode_attention(None, 0, 1, None, None, None, 0, None, 0.1, None, 0, None, None) == osc.ERR_INVALID_ARG
    assert lib.oscar_cache_destroy(None) == 0


@pytest.mark.parametrize("head", [0, 1])
def test_host_calibration_matches_oracle(osc, head):
    qc, kc, vc = synth.calibration(50, 0, head)
    sm = float(np.float32(synth.sm_scale()))      # the ABI passes sm_scale as float32
    got = osc.calibrate(qc, kc, vc, sm)
    ref = rotation.calibrate(qc, kc, vc, sm)
    # eigenvalues are unique; eigenvectors are unique up to the sign convention both sides fix
    assert np.abs(got["eig_K"] - ref["eig_Q"]).max() <= 1e-9 * ref["eig_Q"][0]
    assert np.abs(got["eig_V"] - ref["eig_S"]).max() <= 1e-9 * ref["eig_S"][0]
    assert np.abs(got["U_K"] - ref["U_K"]).max() < 1e-5
    assert np.abs(got["U_V"] - ref["U_V"]).max() < 1e-4
    assert np.abs(got["tau_K"] - ref["tau_K"]).max() <= 1e-5 * np.abs(ref["tau_K"]).max()
    assert np.abs(got["tau_V"] - ref["tau_V"]).max() <= 1e-4 * np.abs(ref["tau_V"]).max()


@pytest.mark.parametrize("head", [0, 1])
def test_host_codebook_calibration_matches_oracle(osc, head):
    from oracle import codebook as CB
    from oracle import pool as P
    qc, kc, vc = synth.calibration(51, 0, head)
    cal = rotation.calibrate(qc, kc, vc, synth.sm_scale())
    xk = P.rotated_f32(kc, cal["U_K"].astype(np.float32))
    tk = cal["tau_K"].astype(np.float32)
    got = osc.calibrate_codebook(xk, tk)
    ref = CB.calibrate_codebook(xk, tk)
    assert np.array_equal(got, ref), (got, ref)
    # heavy-tailed rows with clipping and constant groups mixed in
    rng = np.random.default_rng(7 + head)
    x = (rng.standard_t(3, size=(3000, 128)) * rng.uniform(0.1, 3.0, size=(3000, 1))).astype(np.float32)
    x[::17, :64] = 0.5
    tau = rng.uniform(0.5, 4.0, 128).astype(np.float32)
    assert np.array_equal(osc.calibrate_codebook(x, tau), CB.calibrate_codebook(x, tau))


def test_codebook_layout_and_argument_checks(osc):
    rc, pb, _ = _bytes(osc, meta_format=2)
    rc0, pb0, _ = _bytes(osc, meta_format=0)
    assert rc == 0 and pb == pb0                   # same blocks as the fp16 format
    lib = osc.lib()
    assert lib.oscar_set_codebook(None, 0, None, None, None) == osc.ERR_INVALID_ARG
    assert lib.oscar_calibrate_codebook(None, 1, None, None) == osc.ERR_INVALID_ARG
