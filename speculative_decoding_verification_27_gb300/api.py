"""Python binding of libspecverify.so, with the C ABI's names.

Argument marshalling only: every step runs in the library's CUDA kernels.
Tensors must be CUDA tensors; there is no CPU path, and a missing library is an
error, not a fallback. PyTorch supplies device memory and the current stream.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

from .build import LIB_PATH, ROOT

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_CUDA, SV_ERR_TIMEOUT, SV_ERR_UNIMPLEMENTED, SV_ERR_DATA = range(6)
SV_FP32, SV_BF16 = 0, 1
SV_MODE_SAMPLE, SV_MODE_GREEDY = 0, 1
SV_DATA_BAD_OFFSETS = 0x1
SV_DATA_BAD_TOKEN = 0x2
SV_DATA_EMPTY_ROW = 0x4
SV_DATA_BAD_MODE = 0x8
SV_DATA_DEGENERATE_RESIDUAL = 0x10
SV_DEV_COPY_TIMEOUT = 0x20
SV_ONEHOT_ROW_BYTES_DEFAULT = 128 * 1024  # sv_set_onehot_row_bytes' initial limit

HEADER = os.path.join(ROOT, "include", "spec_verify.h")

_lib = None


class SpecVerifyError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")
        self.status = status


def load() -> ctypes.CDLL:
    """Load the CUDA library (built in-tree by build.build_library())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it first "
            "(speculative_decoding_verification_27_gb300.build.build_library())")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.spec_verify_workspace_size.argtypes = [i32, i32, i32]
    lib.spec_verify_workspace_size.restype = sz
    lib.spec_verify.argtypes = [P, P, ctypes.c_int, i32, i32, P, P, P, P, f32, P, P, P, P, sz, P]
    lib.spec_verify.restype = ctypes.c_int
    lib.spec_verify_greedy.argtypes = [P, ctypes.c_int, i32, i32, P, P, P, P, P, sz, P]
    lib.spec_verify_greedy.restype = ctypes.c_int
    lib.ngram_propose.argtypes = [P, i64, P, i32, i32, i32, i32, P, P, P, P]
    lib.ngram_propose.restype = ctypes.c_int
    lib.sv_pack_drafts.argtypes = [P, P, i32, i32, P, P, P]
    lib.sv_pack_drafts.restype = ctypes.c_int
    lib.sv_check_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32)]
    lib.sv_check_status.restype = ctypes.c_int
    lib.sv_status_string.argtypes = [ctypes.c_int]
    lib.sv_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def header_functions() -> list:
    """Names of the functions declared in include/spec_verify.h."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(\w+)\s*\(", text)) - {"defined", "if"})


def status_string(status: int) -> str:
    return load().sv_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != SV_OK:
        raise SpecVerifyError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("spec_verify tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("spec_verify tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SV_FP32
    if t.dtype == torch.bfloat16:
        return SV_BF16
    raise ValueError("logits must be float32 or bfloat16")


def spec_verify_workspace_size(B: int, R_t: int, V: int) -> int:
    return int(load().spec_verify_workspace_size(int(B), int(R_t), int(V)))


def new_workspace(B: int, R_t: int, V: int, device="cuda") -> torch.Tensor:
    """Zero-filled workspace (the library leaves it zeroed after each call)."""
    return torch.zeros(spec_verify_workspace_size(B, R_t, V), dtype=torch.uint8, device=device)


# Default workspaces, one per (device, stream, entry point): calls on one
# stream run in order and the library leaves its counters at zero after each
# call, so one block serves every call whose workspace layout is the same.
# The layout follows (B, V) for spec_verify / spec_verify_greedy and (B, R_t,
# V) for spec_verify_filtered (its thresholds come first); when it changes,
# or the block is too small, the block is cleared (or grown to the next power
# of two and cleared) before the call. Calls with an unchanged layout clear
# nothing and allocate nothing.
_default_ws: dict = {}
default_workspace_clears = 0   # blocks allocated or cleared so far (each one fill launch)


def default_workspace(nbytes: int, device, stream=None, layout=None) -> torch.Tensor:
    """The cached workspace of `stream` (current stream if None) on `device`
    for calls with workspace layout `layout`, at least `nbytes` long. Calls
    that pass no workspace use it; pass it to sv_check_status to read the
    data-error bits of those calls."""
    dev = torch.device(device)
    idx = dev.index if dev.index is not None else torch.cuda.current_device()
    s = torch.cuda.current_stream(idx) if stream is None else stream
    global default_workspace_clears
    key = (idx, s.cuda_stream, layout[0] if layout else None)
    ent = _default_ws.get(key)
    if ent is None or ent[0].numel() < nbytes:
        default_workspace_clears += 1
        size = 1 << max(12, (int(nbytes) - 1).bit_length())
        with torch.cuda.stream(s):
            ent = [torch.zeros(size, dtype=torch.uint8, device=torch.device("cuda", idx)), layout]
        _default_ws[key] = ent
    elif ent[1] != layout:
        default_workspace_clears += 1
        with torch.cuda.stream(s):
            ent[0].zero_()
        ent[1] = layout
    return ent[0]


def reset_default_workspaces() -> None:
    """Drops the cached workspaces (needed only after SV_DEV_COPY_TIMEOUT,
    which leaves a workspace's counters set)."""
    _default_ws.clear()


def spec_verify(target: torch.Tensor, draft: Optional[torch.Tensor], draft_tokens: torch.Tensor,
                cu_draft: torch.Tensor, uniforms: torch.Tensor, temperature: float,
                mode: Optional[torch.Tensor] = None, *, out_tokens=None, out_len=None,
                out_probs=None, want_probs: bool = True, workspace=None, stream=None):
    """Lossless verify-and-commit. Returns (out_tokens, out_len, out_probs)."""
    lib = load()
    B = cu_draft.shape[0] - 1
    R_t = target.shape[0]
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.full((R_t,), -1, dtype=torch.int32, device=dev)
    if out_len is None:
        out_len = torch.zeros(B, dtype=torch.int32, device=dev)
    if out_probs is None and want_probs:
        out_probs = torch.empty((R_t, 2), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = default_workspace(spec_verify_workspace_size(B, R_t, target.shape[1]), dev, stream,
                                      ("verify", B, target.shape[1]))
    st = lib.spec_verify(_ptr(target), _ptr(draft), _dtype(target), int(target.shape[1]), int(B),
                         _ptr(draft_tokens), _ptr(cu_draft), _ptr(mode), _ptr(uniforms),
                         float(temperature), _ptr(out_tokens), _ptr(out_len), _ptr(out_probs),
                         _ptr(workspace), workspace.numel(), _stream(stream))
    _check("spec_verify", st)
    return out_tokens, out_len, out_probs


SV_NOALLOC_SCRATCH_BYTES = 4 << 20


def _noalloc_fn():
    lib = load()
    fn = lib.spec_verify_noalloc
    P = ctypes.c_void_p
    fn.argtypes = [P, P, ctypes.c_int, ctypes.c_int32, ctypes.c_int32, P, P, P, P, ctypes.c_float,
                   P, P, P, P, P]
    fn.restype = ctypes.c_int
    return fn


def spec_verify_noalloc(target: torch.Tensor, draft: Optional[torch.Tensor], draft_tokens: torch.Tensor,
                        cu_draft: torch.Tensor, uniforms: torch.Tensor, temperature: float,
                        mode: Optional[torch.Tensor], out_tokens: torch.Tensor, out_len: torch.Tensor,
                        out_probs: Optional[torch.Tensor] = None,
                        status_out: Optional[torch.Tensor] = None, stream=None):
    """spec_verify on the library's fixed scratch block: no workspace argument
    and no allocation. Outputs are the caller's. Calls on one device must not
    overlap.

    status_out: a one-element int32 CUDA tensor that receives the call's
    SV_DATA_* / SV_DEV_* bits (0 = clean). With None the bits are dropped:
    a call with bad device data (offsets, tokens) then raises nothing and its
    outputs are unspecified, and the block's own status word cannot be read
    afterwards. Pass one whenever the inputs are not known to be valid."""
    B = cu_draft.shape[0] - 1
    st = _noalloc_fn()(_ptr(target), _ptr(draft), _dtype(target), int(target.shape[1]), int(B),
                       _ptr(draft_tokens), _ptr(cu_draft), _ptr(mode), _ptr(uniforms),
                       float(temperature), _ptr(out_tokens), _ptr(out_len), _ptr(out_probs),
                       _ptr(status_out), _stream(stream))
    _check("spec_verify_noalloc", st)
    return out_tokens, out_len, out_probs


def spec_verify_greedy(target: torch.Tensor, draft_tokens: torch.Tensor, cu_draft: torch.Tensor, *,
                       out_tokens=None, out_len=None, workspace=None, stream=None):
    """Strict (greedy) verify-and-commit. Returns (out_tokens, out_len)."""
    lib = load()
    B = cu_draft.shape[0] - 1
    R_t = target.shape[0]
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.full((R_t,), -1, dtype=torch.int32, device=dev)
    if out_len is None:
        out_len = torch.zeros(B, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = default_workspace(spec_verify_workspace_size(B, R_t, target.shape[1]), dev, stream,
                                      ("verify", B, target.shape[1]))
    st = lib.spec_verify_greedy(_ptr(target), _dtype(target), int(target.shape[1]), int(B),
                                _ptr(draft_tokens), _ptr(cu_draft), _ptr(out_tokens), _ptr(out_len),
                                _ptr(workspace), workspace.numel(), _stream(stream))
    _check("spec_verify_greedy", st)
    return out_tokens, out_len


def ngram_propose(histories: torch.Tensor, hist_len: torch.Tensor, min_n: int, max_n: int,
                  max_tokens: int, *, out_tokens=None, out_count=None, out_n=None, stream=None):
    """N-gram / prompt-lookup proposer. Returns (out_tokens [B, max_tokens], out_count, out_n)."""
    lib = load()
    B, stride = histories.shape
    dev = histories.device
    if out_tokens is None:
        out_tokens = torch.empty((B, max_tokens), dtype=torch.int32, device=dev)
    if out_count is None:
        out_count = torch.empty(B, dtype=torch.int32, device=dev)
    if out_n is None:
        out_n = torch.empty(B, dtype=torch.int32, device=dev)
    st = lib.ngram_propose(_ptr(histories), int(stride), _ptr(hist_len), int(B), int(min_n),
                           int(max_n), int(max_tokens), _ptr(out_tokens), _ptr(out_count),
                           _ptr(out_n), _stream(stream))
    _check("ngram_propose", st)
    return out_tokens, out_count, out_n


SV_SUFFIX_MAX_OCC = 256


def suffix_propose(histories: torch.Tensor, hist_len: torch.Tensor, min_n: int, max_n: int,
                   max_tokens: int, min_share: float = 0.5, max_occ: int = SV_SUFFIX_MAX_OCC, *,
                   out_tokens=None, out_count=None, out_n=None, stream=None):
    """Frequency-ranked suffix proposer. Returns (out_tokens [B, max_tokens], out_count, out_n)."""
    lib = load()
    fn = lib.suffix_propose
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [P, ctypes.c_int64, P, i32, i32, i32, i32, ctypes.c_float, i32, P, P, P, P]
    fn.restype = ctypes.c_int
    B, stride = histories.shape
    dev = histories.device
    if out_tokens is None:
        out_tokens = torch.empty((B, max_tokens), dtype=torch.int32, device=dev)
    if out_count is None:
        out_count = torch.empty(B, dtype=torch.int32, device=dev)
    if out_n is None:
        out_n = torch.empty(B, dtype=torch.int32, device=dev)
    st = fn(_ptr(histories), int(stride), _ptr(hist_len), int(B), int(min_n), int(max_n),
            int(max_tokens), float(min_share), int(max_occ), _ptr(out_tokens), _ptr(out_count),
            _ptr(out_n), _stream(stream))
    _check("suffix_propose", st)
    return out_tokens, out_count, out_n


def sv_pack_drafts(tokens: torch.Tensor, counts: torch.Tensor, max_tokens: int, *, cu_draft=None,
                   packed=None, stream=None):
    """(cu_draft [B+1], packed [B*max_tokens]) from padded proposals and their counts."""
    lib = load()
    B = counts.shape[0]
    dev = counts.device
    if cu_draft is None:
        cu_draft = torch.empty(B + 1, dtype=torch.int32, device=dev)
    if packed is None:
        packed = torch.empty(max(B * max_tokens, 1), dtype=torch.int32, device=dev)
    st = lib.sv_pack_drafts(_ptr(tokens), _ptr(counts), int(B), int(max_tokens), _ptr(cu_draft),
                            _ptr(packed), _stream(stream))
    _check("sv_pack_drafts", st)
    return cu_draft, packed


def sv_check_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronize, read and clear the device status word; returns the SV_DATA_* bits."""
    bits = ctypes.c_uint32(0)
    st = load().sv_check_status(_ptr(workspace), _stream(stream), ctypes.byref(bits))
    if st not in (SV_OK, SV_ERR_DATA, SV_ERR_TIMEOUT):
        raise SpecVerifyError("sv_check_status", st)
    return int(bits.value)


# ---------------------------------------------------------------------------
# Acceptance statistics and the draft-length controller
# ---------------------------------------------------------------------------
SV_METRICS_MAX_POS = 32
_METRIC_SCALARS = ("rounds", "rounds_with_draft", "drafted", "accepted", "committed")
_METRIC_WORDS = len(_METRIC_SCALARS) + 3 * SV_METRICS_MAX_POS


def new_metrics(device="cuda") -> torch.Tensor:
    """A zeroed sv_metrics block on the device (64-bit counters)."""
    return torch.zeros(_METRIC_WORDS, dtype=torch.int64, device=device)


def sv_accumulate_metrics(cu_draft: torch.Tensor, out_len: torch.Tensor, metrics: torch.Tensor,
                          stream=None) -> torch.Tensor:
    """Adds one verify call's rounds to `metrics` (see new_metrics)."""
    lib = load()
    fn = lib.sv_accumulate_metrics
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    if metrics.numel() != _METRIC_WORDS or metrics.dtype != torch.int64:
        raise ValueError("metrics must come from new_metrics()")
    _check("sv_accumulate_metrics", fn(_ptr(cu_draft), _ptr(out_len), int(out_len.numel()),
                                       _ptr(metrics), _stream(stream)))
    return metrics


def metrics_dict(metrics: torch.Tensor) -> dict:
    """The counters as a host dict (keys as in the header's sv_metrics)."""
    v = [int(x) for x in metrics.cpu().tolist()]
    d = dict(zip(_METRIC_SCALARS, v[:5]))
    P = SV_METRICS_MAX_POS
    d["offered"], d["reached"], d["accepted_at"] = v[5:5 + P], v[5 + P:5 + 2 * P], v[5 + 2 * P:5 + 3 * P]
    return d


class _Adapt(ctypes.Structure):
    _fields_ = [("window", ctypes.c_int32), ("min_k", ctypes.c_int32), ("max_k", ctypes.c_int32),
                ("k", ctypes.c_int32), ("count", ctypes.c_int32), ("next", ctypes.c_int32),
                ("target", ctypes.c_double), ("ratio", ctypes.c_double * 1024)]


class AdaptiveDraftLength:
    """The library's sliding-window draft-length controller (host code)."""

    def __init__(self, window=100, min_k=1, max_k=10, target=0.7, initial_k=5):
        lib = load()
        lib.sv_adapt_init.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_double, ctypes.c_int32]
        lib.sv_adapt_init.restype = ctypes.c_int
        lib.sv_adapt_update.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32]
        lib.sv_adapt_update.restype = ctypes.c_int
        lib.sv_adapt_draft_length.argtypes = [ctypes.c_void_p]
        lib.sv_adapt_draft_length.restype = ctypes.c_int32
        self._lib = lib
        self._s = _Adapt()
        _check("sv_adapt_init", lib.sv_adapt_init(ctypes.byref(self._s), window, min_k, max_k,
                                                  float(target), initial_k))

    def update(self, draft_len: int, accepted_len: int) -> int:
        _check("sv_adapt_update", self._lib.sv_adapt_update(ctypes.byref(self._s), draft_len, accepted_len))
        return self.draft_length

    @property
    def draft_length(self) -> int:
        return int(self._lib.sv_adapt_draft_length(ctypes.byref(self._s)))


# ---------------------------------------------------------------------------
# Top-k / top-p filtered verify
# ---------------------------------------------------------------------------
def spec_verify_filtered_workspace_size(B: int, R_t: int, V: int) -> int:
    lib = load()
    lib.spec_verify_filtered_workspace_size.argtypes = [ctypes.c_int32] * 3
    lib.spec_verify_filtered_workspace_size.restype = ctypes.c_size_t
    return int(lib.spec_verify_filtered_workspace_size(int(B), int(R_t), int(V)))


def spec_verify_filtered(target: torch.Tensor, draft: Optional[torch.Tensor], draft_tokens: torch.Tensor,
                         cu_draft: torch.Tensor, uniforms: torch.Tensor, temperature: float,
                         top_k: int = 0, top_p: float = 1.0, mode: Optional[torch.Tensor] = None, *,
                         out_tokens=None, out_len=None, out_probs=None, want_probs: bool = True,
                         workspace=None, stream=None):
    """Verify-and-commit on top-k / top-p filtered distributions.
    Returns (out_tokens, out_len, out_probs)."""
    lib = load()
    fn = lib.spec_verify_filtered
    P = ctypes.c_void_p
    fn.argtypes = [P, P, ctypes.c_int, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P, P, P, P,
                   ctypes.c_float, ctypes.c_int32, ctypes.c_float, P, P, P, P, ctypes.c_size_t, P]
    fn.restype = ctypes.c_int
    B = cu_draft.shape[0] - 1
    R_t = target.shape[0]
    V = target.shape[1]
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.full((R_t,), -1, dtype=torch.int32, device=dev)
    if out_len is None:
        out_len = torch.zeros(B, dtype=torch.int32, device=dev)
    if out_probs is None and want_probs:
        out_probs = torch.empty((R_t, 2), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = default_workspace(spec_verify_filtered_workspace_size(B, R_t, V), dev, stream,
                                      ("filtered", B, R_t, V))
    st = fn(_ptr(target), _ptr(draft), _dtype(target), int(V), int(B), int(R_t), _ptr(draft_tokens),
            _ptr(cu_draft), _ptr(mode), _ptr(uniforms), float(temperature), int(top_k), float(top_p),
            _ptr(out_tokens), _ptr(out_len), _ptr(out_probs), _ptr(workspace), workspace.numel(),
            _stream(stream))
    _check("spec_verify_filtered", st)
    return out_tokens, out_len, out_probs


def sv_set_onehot_row_bytes(nbytes: int) -> int:
    """Largest row (V * element size, in bytes) that spec_verify runs with
    the one-CTA-per-row kernel for one-hot batches (0: never; negative: only
    read); returns the previous limit. Process-wide."""
    lib = load()
    lib.sv_set_onehot_row_bytes.argtypes = [ctypes.c_int32]
    lib.sv_set_onehot_row_bytes.restype = ctypes.c_int32
    return int(lib.sv_set_onehot_row_bytes(int(nbytes)))


def sv_set_cluster_rows(rows: int) -> int:
    """Largest workspace (in target rows) that spec_verify runs with the
    cluster kernel (0: never; negative: only read); returns the previous
    threshold. Process-wide."""
    lib = load()
    lib.sv_set_cluster_rows.argtypes = [ctypes.c_int32]
    lib.sv_set_cluster_rows.restype = ctypes.c_int32
    return int(lib.sv_set_cluster_rows(int(rows)))


SV_SELECT_UNIFORM, SV_SELECT_LONGEST_BIASED = 0, 1


def sv_select_candidates(cu_cand: torch.Tensor, out_len: torch.Tensor, policy: int,
                         u_select: Optional[torch.Tensor] = None, *, best=None, best_len=None,
                         stream=None):
    """Per request, the kept candidate under `policy` (SV_SELECT_UNIFORM needs
    one selection uniform per request in u_select; SV_SELECT_LONGEST_BIASED
    is not distribution-preserving). Returns (best, best_len)."""
    lib = load()
    fn = lib.sv_select_candidates
    P = ctypes.c_void_p
    fn.argtypes = [P, P, ctypes.c_int32, ctypes.c_int32, P, P, P, P]
    fn.restype = ctypes.c_int
    B = cu_cand.shape[0] - 1
    if best is None:
        best = torch.empty(B, dtype=torch.int32, device=cu_cand.device)
    if best_len is None:
        best_len = torch.empty(B, dtype=torch.int32, device=cu_cand.device)
    _check("sv_select_candidates", fn(_ptr(cu_cand), _ptr(out_len), int(B), int(policy), _ptr(u_select),
                                      _ptr(best), _ptr(best_len), _stream(stream)))
    return best, best_len
