"""The C ABI without a GPU: the library builds for sm_103a, loads, exports every
function include/spec_verify.h declares, and rejects bad arguments on the host
before touching CUDA."""
import ctypes
import subprocess

import pytest

from speculative_decoding_verification_27_gb300 import api, build

FAKE = ctypes.c_void_p(0x10000)       # never dereferenced: validation rejects first
MISALIGNED = ctypes.c_void_p(0x10001)


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return api.load()


def test_exports_every_declared_function(lib):
    names = api.header_functions()
    assert {"spec_verify", "spec_verify_greedy", "ngram_propose", "sv_pack_drafts",
            "sv_check_status", "sv_status_string", "spec_verify_workspace_size"} <= set(names)
    exported = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True,
                              text=True, check=True).stdout.split()
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)


def test_workspace_size(lib):
    a16 = lambda x: (x + 15) // 16 * 16
    for B, R, V in [(1, 5, 32000), (64, 384, 128256), (256, 2048, 151936), (513, 3000, 256000), (7, 9, 1)]:
        S = min(B, 4096)            # draw slots
        tiles = (V + 1023) // 1024  # tile sums per slot (fp32-sized tiles)
        split = a16(4 * 4096) + 32 * 16384  # counters and records of split rows
        per_row = 32 + 4 * tiles    # record + fp32 tile sums of a row streamed alone
        want = 64 + a16(8 * B) + a16(4 * S) + 64 * S + a16(8 * S * tiles) + split + per_row * R
        assert api.spec_verify_workspace_size(B, R, V) == want
    assert lib.spec_verify_workspace_size(-1, 4, 10) == 0
    assert lib.spec_verify_workspace_size(4, 4, 0) == 0


def test_status_strings(lib):
    assert api.status_string(0) == "SV_OK"
    assert api.status_string(1) == "SV_ERR_INVALID_ARG"
    assert api.status_string(5) == "SV_ERR_DATA"
    assert api.status_string(99) == "SV_ERR_UNKNOWN"


def _verify(lib, **kw):
    a = dict(target=FAKE, draft=None, dtype=1, V=128, B=2, toks=FAKE, cu=FAKE, mode=None, u=FAKE,
             T=1.0, ot=FAKE, ol=FAKE, op=None, ws=FAKE, wsb=1 << 20, st=None)
    a.update(kw)
    return lib.spec_verify(a["target"], a["draft"], a["dtype"], a["V"], a["B"], a["toks"], a["cu"],
                           a["mode"], a["u"], a["T"], a["ot"], a["ol"], a["op"], a["ws"], a["wsb"],
                           a["st"])


def test_spec_verify_host_validation(lib):
    E = api.SV_ERR_INVALID_ARG
    assert _verify(lib, B=0) == api.SV_OK  # empty batch: nothing to do, nothing launched
    assert _verify(lib, B=-1) == E
    assert _verify(lib, V=0) == E
    assert _verify(lib, V=1 << 20) == E        # beyond the largest vocabulary
    assert _verify(lib, dtype=7) == E
    assert _verify(lib, T=0.0) == E
    assert _verify(lib, T=-1.0) == E
    assert _verify(lib, T=float("nan")) == E
    assert _verify(lib, T=float("inf")) == E
    assert _verify(lib, target=None) == E
    assert _verify(lib, cu=None) == E
    assert _verify(lib, u=None) == E
    assert _verify(lib, ot=None) == E
    assert _verify(lib, ws=None) == E
    assert _verify(lib, target=MISALIGNED) == E   # not element-aligned
    assert _verify(lib, ws=MISALIGNED) == E
    assert _verify(lib, wsb=16) == E               # smaller than the header
    # Strict mode needs neither a temperature nor uniforms.
    assert lib.spec_verify_greedy(FAKE, 1, 0, 2, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == E
    assert lib.spec_verify_greedy(FAKE, 1, 16, 0, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == api.SV_OK


def test_ngram_and_pack_host_validation(lib):
    E = api.SV_ERR_INVALID_ARG
    ng = lambda B=2, mn=1, mx=3, mt=5, stride=16: lib.ngram_propose(FAKE, stride, FAKE, B, mn, mx, mt, FAKE, FAKE, FAKE, None)
    assert ng(B=0) == api.SV_OK
    assert ng(B=-1) == E
    assert ng(mn=0) == E
    assert ng(mn=3, mx=2) == E
    assert ng(mt=-1) == E
    assert ng(stride=-1) == E
    assert lib.ngram_propose(MISALIGNED, 16, FAKE, 2, 1, 3, 5, FAKE, FAKE, FAKE, None) == E
    fn = lib.suffix_propose
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p] + [ctypes.c_int32] * 4 + \
        [ctypes.c_float, ctypes.c_int32] + [ctypes.c_void_p] * 4
    sf = lambda B=2, mn=1, mx=3, mt=5, share=0.5, occ=256, h=FAKE: fn(h, 16, FAKE, B, mn, mx, mt, share, occ,
                                                                     FAKE, FAKE, FAKE, None)
    assert sf(B=0) == api.SV_OK
    assert sf(B=-1) == E
    assert sf(mn=0) == E
    assert sf(mn=3, mx=2) == E
    assert sf(mt=-1) == E
    assert sf(occ=0) == E
    assert sf(occ=257) == E
    assert sf(share=-0.1) == E
    assert sf(share=1.5) == E
    assert sf(share=float("nan")) == E
    assert sf(h=MISALIGNED) == E
    assert lib.sv_pack_drafts(FAKE, FAKE, -1, 5, FAKE, FAKE, None) == E
    assert lib.sv_pack_drafts(FAKE, FAKE, 2, 5, None, FAKE, None) == E
    bits = ctypes.c_uint32(0)
    assert lib.sv_check_status(None, None, ctypes.byref(bits)) == E


def test_python_binding_rejects_host_tensors(lib):
    import torch
    t = torch.zeros((3, 8), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        api.spec_verify_greedy(t, torch.zeros(2, dtype=torch.int32), torch.tensor([0, 2], dtype=torch.int32),
                               out_tokens=torch.zeros(3, dtype=torch.int32),
                               out_len=torch.zeros(1, dtype=torch.int32),
                               workspace=torch.zeros(256, dtype=torch.uint8))


def test_kernel_choice_knobs_round_trip(lib):
    """The process-wide thresholds that pick the cluster kernel and the
    one-hot row kernel are host state: negative values only read them, any
    other value sets them and returns the previous one."""
    assert api.sv_set_cluster_rows(-1) == 64
    assert api.sv_set_onehot_row_bytes(-1) == api.SV_ONEHOT_ROW_BYTES_DEFAULT == 128 * 1024
    try:
        assert api.sv_set_cluster_rows(7) == 64
        assert api.sv_set_cluster_rows(-5) == 7
        assert api.sv_set_onehot_row_bytes(0) == 128 * 1024
        assert api.sv_set_onehot_row_bytes(-1) == 0
    finally:
        api.sv_set_cluster_rows(64)
        api.sv_set_onehot_row_bytes(api.SV_ONEHOT_ROW_BYTES_DEFAULT)
    assert api.sv_set_cluster_rows(-1) == 64 and api.sv_set_onehot_row_bytes(-1) == 128 * 1024


def _filtered(lib, **kw):
    P, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    lib.spec_verify_filtered.argtypes = [P, P, ctypes.c_int, i32, i32, i32, P, P, P, P, f32, i32, f32,
                                         P, P, P, P, ctypes.c_size_t, P]
    lib.spec_verify_filtered.restype = ctypes.c_int
    a = dict(target=FAKE, draft=None, dtype=1, V=128, B=2, R_t=6, toks=FAKE, cu=FAKE, mode=None, u=FAKE,
             T=1.0, k=10, p=0.9, ot=FAKE, ol=FAKE, op=None, ws=FAKE, wsb=1 << 20, st=None)
    a.update(kw)
    return lib.spec_verify_filtered(a["target"], a["draft"], a["dtype"], a["V"], a["B"], a["R_t"], a["toks"],
                                    a["cu"], a["mode"], a["u"], a["T"], a["k"], a["p"], a["ot"], a["ol"],
                                    a["op"], a["ws"], a["wsb"], a["st"])


def test_spec_verify_filtered_host_validation(lib):
    """Every argument the filtered step checks is checked before its first
    kernel: without a GPU a call that got past the checks would fail in
    CUDA (SV_ERR_CUDA), so each rejection here comes first."""
    E = api.SV_ERR_INVALID_ARG
    assert _filtered(lib, B=0) == api.SV_OK
    assert _filtered(lib, k=-1) == E
    assert _filtered(lib, p=0.0) == E
    assert _filtered(lib, R_t=1) == E                 # fewer rows than requests
    assert _filtered(lib, T=0.0) == E
    assert _filtered(lib, ws=None) == E
    assert _filtered(lib, ws=MISALIGNED) == E
    assert _filtered(lib, wsb=64) == E                # smaller than the thresholds' part
    need = int(lib.spec_verify_filtered_workspace_size(2, 6, 128))
    assert need > 0
    assert _filtered(lib, wsb=need - api.spec_verify_workspace_size(2, 6, 128) + 16) == E  # no room for the verify part
    assert _filtered(lib, ot=None) == E               # checked before the thresholds are enqueued
    assert _filtered(lib, ol=None) == E
    assert _filtered(lib, u=None) == E
    assert _filtered(lib, cu=MISALIGNED) == E
    assert _filtered(lib, op=MISALIGNED) == E
