"""ctypes binding of libdomino_gb300.so (include/domino.h), same names as the C ABI.

Argument marshalling only: torch tensors are passed as device pointers, streams
as cudaStream_t handles; every step of the computation runs in the library's
CUDA kernels.  There is no CPU or PyTorch fallback: if the library is missing
or the device is not a GB300, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, List, Optional, Sequence, Tuple

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libdomino_gb300.so")

# enums of include/domino.h
STATUS = {0: "DOMINO_OK", 1: "DOMINO_ERR_INVALID_ARG", 2: "DOMINO_ERR_UNSUPPORTED", 3: "DOMINO_ERR_ALIGNMENT",
          4: "DOMINO_ERR_WORKSPACE", 5: "DOMINO_ERR_CUDA", 6: "DOMINO_ERR_TIMEOUT", 7: "DOMINO_ERR_DEVICE"}
ACT = {"gelu": 0, "gelu_tanh": 1, "swiglu": 2, "identity": 3}
PARTIAL = {"f32": 0, "bf16": 1}
SCHEDULE = {"serial": 0, "streams": 1, "fused": 2}
KERNEL_KIND = {0: "gemm1", 1: "gemm2", 2: "shard_sum", 3: "bwd_dh", 4: "bwd_dx", 5: "bwd_dw", 6: "fused", 7: "attn",
               8: "bwd_dx_fused", 9: "attn_out_fused"}
FLAG_KERNEL_TIMES = 1
FLAG_ONE_CTA = 2
MAX_SHARDS = 16


class DominoError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}: {detail}")


class MlpDesc(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int64),
        ("d", ctypes.c_int64),
        ("F", ctypes.c_int64),
        ("P", ctypes.c_int32),
        ("mu", ctypes.c_int32),
        ("out_slices", ctypes.c_int32),
        ("act", ctypes.c_int32),
        ("partial_dtype", ctypes.c_int32),
        ("schedule", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
        ("reserve_sms", ctypes.c_int32),
        ("timeout_ns", ctypes.c_uint64),
    ]


class Timeline(ctypes.Structure):
    _fields_ = [("start_ns", ctypes.c_uint64), ("gemm_end_ns", ctypes.c_uint64), ("reduce_end_ns", ctypes.c_uint64)]


class KernelTime(ctypes.Structure):
    _fields_ = [
        ("call", ctypes.c_int32),
        ("kind", ctypes.c_int32),
        ("chunk", ctypes.c_int32),
        ("slice", ctypes.c_int32),
        ("stream", ctypes.c_int32),
        ("start_ms", ctypes.c_float),
        ("end_ms", ctypes.c_float),
    ]


class AttnDesc(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64),
        ("S", ctypes.c_int64),
        ("d", ctypes.c_int64),
        ("H", ctypes.c_int32),
        ("dh", ctypes.c_int32),
        ("P", ctypes.c_int32),
        ("mu", ctypes.c_int32),
        ("partial_dtype", ctypes.c_int32),
        ("schedule", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
        ("reserved", ctypes.c_uint32),
        ("timeout_ns", ctypes.c_uint64),
    ]


class PlanHw(ctypes.Structure):
    _fields_ = [("num_sms", ctypes.c_int32), ("fused_available", ctypes.c_int32), ("l2_bytes", ctypes.c_int64)]


class Plan(ctypes.Structure):
    _fields_ = [
        ("mu", ctypes.c_int32),
        ("schedule", ctypes.c_int32),
        ("reason", ctypes.c_int32),
        ("gemm1_tiles_per_chunk", ctypes.c_int32),
        ("chunk_h_bytes", ctypes.c_int64),
        ("l2_budget_bytes", ctypes.c_int64),
    ]


PLAN_REASON = {0: "fits_l2", 1: "largest_filling", 2: "small"}


class TensorPeak(ctypes.Structure):
    _fields_ = [
        ("tflops", ctypes.c_double),
        ("flops", ctypes.c_double),
        ("ms", ctypes.c_double),
        ("sm_mhz", ctypes.c_double),
        ("flops_per_clk_sm", ctypes.c_double),
        ("clusters", ctypes.c_int32),
        ("num_sms", ctypes.c_int32),
    ]


TENSOR_PEAK_MAX_MMAS = 1 << 22
TENSOR_PEAK_WS_BYTES = 256

_LIB: Optional[ctypes.CDLL] = None
_VP = ctypes.c_void_p
_VPP = ctypes.POINTER(ctypes.c_void_p)

# (name, restype, argtypes) for every entry point of include/domino.h
SIGNATURES = [
    ("domino_mlp_workspace_size", ctypes.c_size_t, [ctypes.POINTER(MlpDesc), ctypes.c_int32]),
    ("domino_mlp_saved_size", ctypes.c_size_t, [ctypes.POINTER(MlpDesc)]),
    ("domino_mlp_fwd", ctypes.c_int, [ctypes.POINTER(MlpDesc), _VP, _VPP, _VPP, _VP, _VP, _VP, ctypes.c_size_t, _VP]),
    ("domino_mlp_fwd_partials", ctypes.c_int,
     [ctypes.POINTER(MlpDesc), _VP, _VPP, _VPP, _VPP, _VPP, _VP, _VP, ctypes.c_size_t, _VP]),
    ("domino_mlp_bwd", ctypes.c_int,
     [ctypes.POINTER(MlpDesc), _VP, _VPP, _VPP, _VP, _VP, _VP, _VPP, _VPP, _VP, ctypes.c_size_t, _VP]),
    ("domino_shard_sum", ctypes.c_int,
     [_VPP, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _VP, ctypes.c_int64, _VP]),
    ("domino_query_device_status", ctypes.c_int, [_VP, _VP]),
    ("domino_read_timeline", ctypes.c_int, [_VP, _VP, ctypes.POINTER(Timeline)]),
    ("domino_selftest_wait_timeout", ctypes.c_int, [_VP, ctypes.c_uint64, _VP]),
    ("domino_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("domino_last_error", ctypes.c_char_p, []),
    ("domino_mlp_fwd_noalloc", ctypes.c_int, [ctypes.POINTER(MlpDesc), _VP, _VPP, _VPP, _VP, _VP]),
    ("domino_mlp_fwd_noalloc_status", ctypes.c_int, [_VP, _VPP]),
    ("domino_kernel_times", ctypes.c_int32, [ctypes.POINTER(KernelTime), ctypes.c_int32]),
    ("domino_kernel_times_reset", None, []),
    ("domino_mlp_plan", ctypes.c_int, [ctypes.POINTER(MlpDesc), ctypes.POINTER(PlanHw), ctypes.POINTER(Plan)]),
    ("domino_attn_plan", ctypes.c_int, [ctypes.POINTER(AttnDesc), ctypes.POINTER(PlanHw), ctypes.POINTER(Plan)]),
    ("domino_mlp_interleaved_workspace_size", ctypes.c_size_t, [ctypes.POINTER(MlpDesc)]),
    ("domino_attn_workspace_size", ctypes.c_size_t, [ctypes.POINTER(AttnDesc)]),
    ("domino_attn_fwd", ctypes.c_int, [ctypes.POINTER(AttnDesc), _VP, _VPP, _VPP, _VP, _VP, ctypes.c_size_t, _VP]),
    ("domino_mlp_fwd_bwd_interleaved", ctypes.c_int,
     [ctypes.POINTER(MlpDesc), _VPP, _VPP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VPP, _VPP, _VP, ctypes.c_size_t, _VP]),
    ("domino_tensor_peak", ctypes.c_int,
     [ctypes.c_int64, ctypes.c_int32, _VP, ctypes.c_size_t, ctypes.c_uint64, _VP, ctypes.POINTER(TensorPeak)]),
]


def lib() -> ctypes.CDLL:
    """Loads the library (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        path = os.environ.get("DOMINO_LIB_PATH") or LIB_PATH  # another build of the same library, if given
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                               "(this package has no CPU or PyTorch fallback)")
        handle = ctypes.CDLL(path)
        for name, res, args in SIGNATURES:
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


def _check(status: int, where: str) -> None:
    if status != 0:
        detail = lib().domino_last_error().decode(errors="replace")
        raise DominoError(status, where, detail)


def _ptr_array(ptrs: Sequence[int]):
    arr = (ctypes.c_void_p * max(1, len(ptrs)))()
    for i, p in enumerate(ptrs):
        arr[i] = p
    return arr


def make_desc(M: int, d: int, F: int, P: int, mu: int, act: str, partial: str, out_slices: int = 1,
              schedule: str = "streams", kernel_times: bool = False, timeout_ns: int = 0,
              pair_cta: bool = True, reserve_sms: int = 0) -> MlpDesc:
    """pair_cta: run the separate-launch GEMMs as paired-CTA 256x256 tiles (default) or,
    if False, as one-CTA 128x256 tiles.  reserve_sms: SMs the library's kernels leave free."""
    flags = (FLAG_KERNEL_TIMES if kernel_times else 0) | (0 if pair_cta else FLAG_ONE_CTA)
    return MlpDesc(M=M, d=d, F=F, P=P, mu=mu, out_slices=out_slices, act=ACT[act], partial_dtype=PARTIAL[partial],
                   schedule=SCHEDULE[schedule], flags=flags, reserve_sms=reserve_sms, timeout_ns=timeout_ns)


def workspace_size(desc: MlpDesc, with_bwd: bool = False) -> int:
    return int(lib().domino_mlp_workspace_size(ctypes.byref(desc), 1 if with_bwd else 0))


def saved_size(desc: MlpDesc) -> int:
    return int(lib().domino_mlp_saved_size(ctypes.byref(desc)))


# ------------------------------------------------------------------ torch side

def _torch():
    import torch
    return torch


def _stream_handle(stream) -> int:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


_WS_CACHE: Dict[Tuple[int, int], object] = {}


def _workspace(nbytes: int, device):
    """A cached uint8 device buffer of at least nbytes (256-byte aligned by torch)."""
    torch = _torch()
    dev = torch.device(device)
    key = (dev.index if dev.index is not None else torch.cuda.current_device(), nbytes)
    buf = _WS_CACHE.get(key)
    if buf is None:
        buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=dev)
        _WS_CACHE[key] = buf
    return buf


def shard_weights(A, B, P: int):
    """Splits mathematical-layout weights into the ABI's per-shard layout.

    A: [d, F] (or a pair (Wg, Wu), each [d, F]); B: [F, d].  Returns
    (A_shards, B_shards): A_shards[p] = A[:, cols_p]^T ([F/P, d]; SwiGLU:
    Wg[:, cols_p]^T stacked over Wu[:, cols_p]^T, [2F/P, d]) and
    B_shards[p] = B[cols_p, :]^T ([d, F/P]), each contiguous.  A one-time
    parameter re-layout (like loading a checkpoint into a tensor-parallel
    layout), not part of the forward pass.
    """
    torch = _torch()
    if isinstance(A, (tuple, list)):
        Wg, Wu = A
        F = Wg.shape[1]
    else:
        Wg, Wu = A, None
        F = A.shape[1]
    Fp = F // P
    A_sh, B_sh = [], []
    for p in range(P):
        cols = slice(p * Fp, (p + 1) * Fp)
        if Wu is not None:
            A_sh.append(torch.cat([Wg[:, cols].t(), Wu[:, cols].t()], dim=0).contiguous())
        else:
            A_sh.append(Wg[:, cols].t().contiguous())
        B_sh.append(B[cols, :].t().contiguous())
    return A_sh, B_sh


def mlp_fwd(X, A_shards: List, B_shards: List, *, F: int, mu: int, act: str, partial: str, out_slices: int = 1,
            schedule: str = "streams", Y=None, saved=None, workspace=None, stream=None, kernel_times: bool = False,
            timeout_ns: int = 0, pair_cta: bool = True, reserve_sms: int = 0):
    """domino_mlp_fwd on torch tensors; returns Y [M, d] bf16."""
    torch = _torch()
    M, d = X.shape
    P = len(A_shards)
    desc = make_desc(M, d, F, P, mu, act, partial, out_slices, schedule, kernel_times, timeout_ns, pair_cta,
                     reserve_sms=reserve_sms)
    if Y is None:
        Y = torch.empty((M, d), dtype=torch.bfloat16, device=X.device)
    need = workspace_size(desc)
    if need == 0:
        _check(lib().domino_mlp_fwd(ctypes.byref(desc), None, None, None, None, None, None, 0, None), "domino_mlp_fwd")
    if workspace is None:
        workspace = _workspace(need, X.device)
    st = lib().domino_mlp_fwd(
        ctypes.byref(desc), X.data_ptr(), _ptr_array([a.data_ptr() for a in A_shards]),
        _ptr_array([b.data_ptr() for b in B_shards]), Y.data_ptr(), saved.data_ptr() if saved is not None else None,
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, "domino_mlp_fwd")
    return Y


def mlp_fwd_partials(X, A_shards: List, B_shards: List, *, F: int, mu: int, act: str, partial: str,
                     out_slices: int = 1, schedule: str = "streams", Z_shards=None, piece_events=None, saved=None,
                     workspace=None, stream=None, kernel_times: bool = False, timeout_ns: int = 0,
                     pair_cta: bool = True, reserve_sms: int = 0):
    """domino_mlp_fwd_partials on torch tensors: the row-parallel partials of every shard, not summed.
    Returns Z_shards (P tensors [M, d], fp32 or bf16 as `partial`).  piece_events: None or mu * out_slices
    torch.cuda.Event objects, each recorded when its (chunk, slice) piece of every partial is written."""
    torch = _torch()
    M, d = X.shape
    P = len(A_shards)
    desc = make_desc(M, d, F, P, mu, act, partial, out_slices, schedule, kernel_times, timeout_ns, pair_cta,
                     reserve_sms=reserve_sms)
    if Z_shards is None:
        dt = torch.float32 if partial == "f32" else torch.bfloat16
        Z_shards = [torch.empty((M, d), dtype=dt, device=X.device) for _ in range(P)]
    need = workspace_size(desc)
    if workspace is None:
        workspace = _workspace(max(need, 256), X.device)
    events = None
    if piece_events is not None:
        for e in piece_events:  # torch creates the CUDA event lazily, on first record
            if e.cuda_event == 0:
                e.record()
        events = _ptr_array([e.cuda_event for e in piece_events])
    st = lib().domino_mlp_fwd_partials(
        ctypes.byref(desc), X.data_ptr(), _ptr_array([a.data_ptr() for a in A_shards]),
        _ptr_array([b.data_ptr() for b in B_shards]), _ptr_array([z.data_ptr() for z in Z_shards]), events,
        saved.data_ptr() if saved is not None else None, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, "domino_mlp_fwd_partials")
    return Z_shards


def mlp_bwd(X, A_shards: List, B_shards: List, dY, saved, *, F: int, mu: int, act: str, partial: str,
            out_slices: int = 1, schedule: str = "streams", dX=None, dA_shards=None, dB_shards=None, workspace=None,
            stream=None, kernel_times: bool = False, timeout_ns: int = 0, pair_cta: bool = True, reserve_sms: int = 0):
    """domino_mlp_bwd on torch tensors; returns (dX, dA_shards, dB_shards).

    `saved` must be the buffer a domino_mlp_fwd call with the same inputs filled."""
    torch = _torch()
    M, d = X.shape
    P = len(A_shards)
    desc = make_desc(M, d, F, P, mu, act, partial, out_slices, schedule, kernel_times, timeout_ns, pair_cta,
                     reserve_sms=reserve_sms)
    if dX is None:
        dX = torch.empty((M, d), dtype=torch.bfloat16, device=X.device)
    if dA_shards is None:
        dA_shards = [torch.empty_like(a) for a in A_shards]
    if dB_shards is None:
        dB_shards = [torch.empty_like(b) for b in B_shards]
    if workspace is None:
        workspace = _workspace(max(workspace_size(desc, with_bwd=True), 256), X.device)
    st = lib().domino_mlp_bwd(
        ctypes.byref(desc), X.data_ptr(), _ptr_array([a.data_ptr() for a in A_shards]),
        _ptr_array([b.data_ptr() for b in B_shards]), dY.data_ptr(), saved.data_ptr(), dX.data_ptr(),
        _ptr_array([a.data_ptr() for a in dA_shards]), _ptr_array([b.data_ptr() for b in dB_shards]),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, "domino_mlp_bwd")
    return dX, dA_shards, dB_shards


def make_attn_desc(B: int, S: int, d: int, H: int, P: int, mu: int, partial: str, schedule: str = "streams",
                   dh: int = 128, kernel_times: bool = False, timeout_ns: int = 0, pair_cta: bool = True) -> AttnDesc:
    flags = (FLAG_KERNEL_TIMES if kernel_times else 0) | (0 if pair_cta else FLAG_ONE_CTA)
    return AttnDesc(B=B, S=S, d=d, H=H, dh=dh, P=P, mu=mu, partial_dtype=PARTIAL[partial],
                    schedule=SCHEDULE[schedule], flags=flags, reserved=0, timeout_ns=timeout_ns)


def attn_workspace_size(desc: AttnDesc) -> int:
    return int(lib().domino_attn_workspace_size(ctypes.byref(desc)))


def shard_attn_weights(Wqkv, Wo, H: int, P: int):
    """Splits mathematical-layout attention weights into the ABI's per-shard layout.

    Wqkv: [d, 3 H dh] (query heads, then key heads, then value heads); Wo: [H dh, d].
    Returns (Wqkv_shards, Wo_shards): Wqkv_shards[p] = [3 Hp dh, d], shard p's query,
    key and value heads' columns of Wqkv transposed; Wo_shards[p] = Wo[rows_p, :]^T
    [d, Hp dh]; each contiguous.  A one-time parameter re-layout."""
    torch = _torch()
    d, n = Wqkv.shape
    dh = n // (3 * H)
    Hp = H // P
    w = Hp * dh
    qkv_sh, o_sh = [], []
    for p in range(P):
        cols = [Wqkv[:, j * H * dh + p * w: j * H * dh + (p + 1) * w] for j in range(3)]
        qkv_sh.append(torch.cat(cols, dim=1).t().contiguous())
        o_sh.append(Wo[p * w:(p + 1) * w, :].t().contiguous())
    return qkv_sh, o_sh


def attn_fwd(X, Wqkv_shards: List, Wo_shards: List, *, S: int, H: int, mu: int, partial: str,
             schedule: str = "streams", Y=None, workspace=None, stream=None, kernel_times: bool = False,
             timeout_ns: int = 0, pair_cta: bool = True):
    """domino_attn_fwd on torch tensors; returns Y [B S, d] bf16."""
    torch = _torch()
    M, d = X.shape
    P = len(Wqkv_shards)
    desc = make_attn_desc(M // S, S, d, H, P, mu, partial, schedule, 128, kernel_times, timeout_ns, pair_cta)
    if Y is None:
        Y = torch.empty((M, d), dtype=torch.bfloat16, device=X.device)
    if workspace is None:
        workspace = _workspace(max(attn_workspace_size(desc), 256), X.device)
    st = lib().domino_attn_fwd(ctypes.byref(desc), X.data_ptr(), _ptr_array([w.data_ptr() for w in Wqkv_shards]),
                               _ptr_array([w.data_ptr() for w in Wo_shards]), Y.data_ptr(), workspace.data_ptr(),
                               workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, "domino_attn_fwd")
    return Y


def interleaved_workspace_size(desc: MlpDesc) -> int:
    return int(lib().domino_mlp_interleaved_workspace_size(ctypes.byref(desc)))


def mlp_fwd_bwd_interleaved(A_shards: List, B_shards: List, Xa, Xb, dYb, saved_b, *, F: int, mu: int, act: str,
                            partial: str, out_slices: int = 1, schedule: str = "streams", Ya=None, saved_a=None,
                            dXb=None, dA_shards=None, dB_shards=None, workspace=None, stream=None,
                            kernel_times: bool = False, timeout_ns: int = 0, pair_cta: bool = True):
    """domino_mlp_fwd_bwd_interleaved: the forward of strand a (Xa -> Ya, saved_a) and the backward
    of strand b (Xb, dYb, saved_b -> dXb, dA_shards, dB_shards) in one call; returns
    (Ya, dXb, dA_shards, dB_shards)."""
    torch = _torch()
    M, d = Xa.shape
    P = len(A_shards)
    desc = make_desc(M, d, F, P, mu, act, partial, out_slices, schedule, kernel_times, timeout_ns, pair_cta)
    if Ya is None:
        Ya = torch.empty((M, d), dtype=torch.bfloat16, device=Xa.device)
    if dXb is None:
        dXb = torch.empty((M, d), dtype=torch.bfloat16, device=Xa.device)
    if dA_shards is None:
        dA_shards = [torch.empty_like(a) for a in A_shards]
    if dB_shards is None:
        dB_shards = [torch.empty_like(x) for x in B_shards]
    if workspace is None:
        workspace = _workspace(max(interleaved_workspace_size(desc), 256), Xa.device)
    st = lib().domino_mlp_fwd_bwd_interleaved(
        ctypes.byref(desc), _ptr_array([a.data_ptr() for a in A_shards]),
        _ptr_array([x.data_ptr() for x in B_shards]), Xa.data_ptr(), Ya.data_ptr(),
        saved_a.data_ptr() if saved_a is not None else None, Xb.data_ptr(), dYb.data_ptr(), saved_b.data_ptr(),
        dXb.data_ptr(), _ptr_array([a.data_ptr() for a in dA_shards]), _ptr_array([x.data_ptr() for x in dB_shards]),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, "domino_mlp_fwd_bwd_interleaved")
    return Ya, dXb, dA_shards, dB_shards


def unshard_grads(dA_shards: List, dB_shards: List, act: str):
    """Inverse of shard_weights for gradients: returns (dA or (dWg, dWu), dB) in
    the mathematical layout ([d, F] and [F, d])."""
    torch = _torch()
    if act == "swiglu":
        Fp = dA_shards[0].shape[0] // 2
        dWg = torch.cat([a[:Fp].t() for a in dA_shards], dim=1)
        dWu = torch.cat([a[Fp:].t() for a in dA_shards], dim=1)
        dA = (dWg, dWu)
    else:
        dA = torch.cat([a.t() for a in dA_shards], dim=1)
    dB = torch.cat([b.t() for b in dB_shards], dim=0)
    return dA, dB


def mlp_fwd_noalloc(X, A_shards: List, B_shards: List, *, F: int, mu: int, act: str, partial: str,
                    out_slices: int = 1, Y=None, stream=None, timeout_ns: int = 0):
    """domino_mlp_fwd_noalloc: the forward pass with the library's own fixed scratch
    array instead of a workspace, for callers that cannot allocate device memory
    while the layer runs.  Serial schedule; returns Y [M, d] bf16."""
    torch = _torch()
    M, d = X.shape
    P = len(A_shards)
    desc = make_desc(M, d, F, P, mu, act, partial, out_slices, "serial", False, timeout_ns)
    if Y is None:
        Y = torch.empty((M, d), dtype=torch.bfloat16, device=X.device)
    st = lib().domino_mlp_fwd_noalloc(
        ctypes.byref(desc), X.data_ptr(), _ptr_array([a.data_ptr() for a in A_shards]),
        _ptr_array([b.data_ptr() for b in B_shards]), Y.data_ptr(), _stream_handle(stream))
    _check(st, "domino_mlp_fwd_noalloc")
    return Y


def mlp_fwd_noalloc_status(stream=None):
    """domino_mlp_fwd_noalloc_status: synchronises, returns and clears the device status of the last
    no-alloc forward (0 = OK), and the device address of the fixed scratch array's header."""
    header = ctypes.c_void_p()
    st = int(lib().domino_mlp_fwd_noalloc_status(_stream_handle(stream), ctypes.byref(header)))
    return st, int(header.value or 0)


def shard_sum(partials: List, Y, *, stream=None):
    """domino_shard_sum: Y = bf16(sum of the fp32 or bf16 partials)."""
    torch = _torch()
    P = len(partials)
    rows, cols = partials[0].shape
    dt = {torch.float32: 0, torch.bfloat16: 1}[partials[0].dtype]
    st = lib().domino_shard_sum(_ptr_array([z.data_ptr() for z in partials]), P, dt, rows, cols,
                                partials[0].stride(0), Y.data_ptr(), Y.stride(0), _stream_handle(stream))
    _check(st, "domino_shard_sum")
    return Y


def read_timeline(workspace, stream=None) -> dict:
    """domino_read_timeline: device timeline (ns) of the last fused forward call on this workspace."""
    tl = Timeline()
    _check(lib().domino_read_timeline(workspace.data_ptr(), _stream_handle(stream), ctypes.byref(tl)),
           "domino_read_timeline")
    return {"start_ns": tl.start_ns, "gemm_end_ns": tl.gemm_end_ns, "reduce_end_ns": tl.reduce_end_ns}


def selftest_wait_timeout(workspace, timeout_ns: int, stream=None) -> None:
    """Launches a kernel whose bounded wait runs out (a flag nothing sets)."""
    _check(lib().domino_selftest_wait_timeout(workspace.data_ptr(), timeout_ns, _stream_handle(stream)),
           "domino_selftest_wait_timeout")


def query_device_status(workspace, stream=None) -> int:
    """Synchronises, returns and clears the device status word (0 = OK)."""
    return int(lib().domino_query_device_status(workspace.data_ptr(), _stream_handle(stream)))


def plan(M: int, d: int, F: int, P: int, act: str, partial: str, out_slices: int = 1, *, num_sms: int = 0,
         l2_bytes: int = 0, fused_available: int = -1) -> dict:
    """domino_mlp_plan: the number of row chunks and the schedule for this problem.  Hardware
    figures left at 0 (fused_available at -1) are read from the current CUDA device."""
    desc = make_desc(M, d, F, P, 1, act, partial, out_slices)
    hw = PlanHw(num_sms=num_sms, fused_available=fused_available, l2_bytes=l2_bytes)
    out = Plan()
    _check(lib().domino_mlp_plan(ctypes.byref(desc), ctypes.byref(hw), ctypes.byref(out)), "domino_mlp_plan")
    sched = {v: k for k, v in SCHEDULE.items()}[out.schedule]
    return {"mu": out.mu, "schedule": sched, "reason": PLAN_REASON.get(out.reason, out.reason),
            "gemm1_tiles_per_chunk": out.gemm1_tiles_per_chunk, "chunk_h_bytes": out.chunk_h_bytes,
            "l2_budget_bytes": out.l2_budget_bytes}


def plan_attn(B: int, S: int, d: int, H: int, P: int, partial: str, *, dh: int = 128, num_sms: int = 0,
              l2_bytes: int = 0) -> dict:
    """domino_attn_plan: the number of sequence chunks and the schedule for this attention block.
    Hardware figures left at 0 are read from the current CUDA device."""
    desc = make_attn_desc(B, S, d, H, P, 1, partial, dh=dh)
    hw = PlanHw(num_sms=num_sms, fused_available=0, l2_bytes=l2_bytes)
    out = Plan()
    _check(lib().domino_attn_plan(ctypes.byref(desc), ctypes.byref(hw), ctypes.byref(out)), "domino_attn_plan")
    sched = {v: k for k, v in SCHEDULE.items()}[out.schedule]
    return {"mu": out.mu, "schedule": sched, "reason": PLAN_REASON.get(out.reason, out.reason),
            "proj_tiles_per_chunk": out.gemm1_tiles_per_chunk, "chunk_qkv_bytes": out.chunk_h_bytes,
            "l2_budget_bytes": out.l2_budget_bytes}


def tensor_peak(mmas_per_cluster: int = 1 << 18, clusters: int = 0, *, workspace=None, stream=None,
                timeout_ns: int = 0) -> dict:
    """domino_tensor_peak: dense bf16 rate of back-to-back paired tcgen05 MMAs on every
    co-resident 2-CTA cluster (clusters=0), with the SM clock measured in the kernel."""
    import torch
    ws = workspace if workspace is not None else torch.zeros(TENSOR_PEAK_WS_BYTES, dtype=torch.uint8, device="cuda")
    s = stream if stream is not None else torch.cuda.current_stream()
    out = TensorPeak()
    _check(lib().domino_tensor_peak(mmas_per_cluster, clusters, ws.data_ptr(), ws.numel(), timeout_ns,
                                    s.cuda_stream, ctypes.byref(out)), "domino_tensor_peak")
    return {"tflops": out.tflops, "flops": out.flops, "ms": out.ms, "sm_mhz": out.sm_mhz,
            "flops_per_clk_sm": out.flops_per_clk_sm, "clusters": out.clusters, "num_sms": out.num_sms}


def kernel_times_reset() -> None:
    lib().domino_kernel_times_reset()


def kernel_times() -> List[dict]:
    """Per-launch event times logged by calls made with kernel_times=True since the last reset."""
    n = lib().domino_kernel_times(None, 0)
    if n <= 0:
        return []
    buf = (KernelTime * n)()
    n = lib().domino_kernel_times(buf, n)
    if n < 0:
        raise DominoError(5, "domino_kernel_times", "event synchronisation failed")
    return [{"call": r.call, "kind": KERNEL_KIND.get(r.kind, r.kind), "chunk": r.chunk, "slice": r.slice,
             "stream": r.stream, "start_ms": r.start_ms, "end_ms": r.end_ms} for r in buf[:n]]
