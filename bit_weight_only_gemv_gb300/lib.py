"""ctypes binding of libw4a16.so (argument marshalling only).

Every function takes torch tensors that already live on the GPU, checks
dtypes/shapes, and passes raw pointers, sizes and the current CUDA stream to
the C ABI declared in include/w4a16.h.  No arithmetic of the method happens
here, and there is no fallback: if the library is missing, ``load()`` raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libw4a16.so")

W4_FLAG_PDL = 1
W4_FLAG_CUDA_CORES = 2
W4_FLAG_TENSOR_CORES = 4
W4_FLAG_SILU_MUL = 8
W4_FLAG_IDS_FINAL = 16


def _id_flags(pdl: bool, ids_final: bool) -> int:
    """ids_final: the ids were written before the previous kernel began
    (W4_FLAG_IDS_FINAL; only meaningful with pdl)."""
    return (W4_FLAG_PDL if pdl else 0) | (W4_FLAG_IDS_FINAL if ids_final else 0)
_PATH_FLAGS = {None: 0, "cuda": W4_FLAG_CUDA_CORES, "tensor": W4_FLAG_TENSOR_CORES}
STATUS = {0: "W4_OK", 1: "W4_ERR_ARG", 2: "W4_ERR_ALIGN", 3: "W4_ERR_SHAPE",
          4: "W4_ERR_WORKSPACE", 5: "W4_ERR_LAUNCH", 6: "W4_ERR_INDEX", 7: "W4_ERR_VALUE",
          8: "W4_ERR_TIMEOUT", 9: "W4_ERR_DEVICE", 10: "W4_ERR_STATE", 11: "W4_ERR_OWNER"}
STATUS_CODE = {v: k for k, v in STATUS.items()}

EXPORTS = ("w4_status_str", "w4_abi_version", "w4_last_cuda_error", "w4a16_gemv", "w4a16_gemv_workspace_bytes", "w4a16_gemv_workspace_bytes_flags",
           "w4a16_gemv_id", "w4a16_gemv_id_scaled", "w4_embed_gather", "w4_pack", "w4_quantize",
           "w4_slot_pool_create", "w4_slot_pool_destroy", "w4_slot_pool_remap",
           "w4_slot_pool_stage", "w4_slot_pool_stats", "w4a16_gemv_plan",
           "w4a16_gemv_static_scratch", "w4_dev_pool_state_bytes", "w4_dev_pool_init",
           "w4_dev_pool_stage", "w4_dev_pool_stats", "w4a16_gemv_chain",
           "w4a16_gemv_chain_workspace_bytes", "w4a16_gemv_chain_plan",
           "w4a16_gemv_chain_task_plan", "w4a16_gemv_id_plan", "w4a16_gemv_prefetch_l2",
           "w4a16_gemv_plan_flags")
W4_TASK_SILU_MUL = 1
W4_MAX_L2_RANGES = 4
CHAIN_MAX_TASKS = 320


class W4Error(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        self.name = STATUS.get(code, str(code))
        super().__init__(f"{what}: {self.name}")


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("path", "ctas", "slices", "threads", "team",
                                            "unit_rows", "chunk_groups", "rows_per_lane",
                                            "smem_bytes", "rows_per_call", "chunk_steps",
                                            "stages", "ctas_per_sm", "tmpl_team",
                                            "tmpl_chunk", "dynamic_windows")]


class GemvTask(ctypes.Structure):
    """struct w4_gemv_task of include/w4a16.h."""
    _fields_ = [("y", ctypes.c_void_p), ("qw", ctypes.c_void_p), ("st", ctypes.c_void_p),
                ("x", ctypes.c_void_p), ("ids", ctypes.c_void_p), ("qw_stride", ctypes.c_size_t),
                ("st_stride", ctypes.c_size_t), ("num_experts", ctypes.c_int),
                ("n_ids", ctypes.c_int), ("x_rows", ctypes.c_int), ("N", ctypes.c_int),
                ("K", ctypes.c_int), ("dep", ctypes.c_int), ("flags", ctypes.c_uint)]


class L2Range(ctypes.Structure):
    """struct w4_l2_range of include/w4a16.h."""
    _fields_ = [("ptr", ctypes.c_void_p), ("bytes", ctypes.c_size_t)]


class ChainPlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("ctas", "threads", "instantiation", "stages",
                                            "stage_bytes", "smem_bytes", "windows")]


class ChainTaskInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("rows_per_window", "rows_per_lane", "team",
                                            "chunk_steps", "chunks", "windows_per_item", "dot")]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library once; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    vp, i32, sz, u32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint
    i32p = ctypes.POINTER(ctypes.c_int32)
    lib.w4_status_str.restype = ctypes.c_char_p
    lib.w4_status_str.argtypes = [i32]
    lib.w4_abi_version.restype = i32
    lib.w4_last_cuda_error.restype = ctypes.c_char_p
    lib.w4_last_cuda_error.argtypes = []
    lib.w4a16_gemv.restype = i32
    lib.w4a16_gemv.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, sz, vp, u32, vp]
    lib.w4a16_gemv_prefetch_l2.restype = i32
    lib.w4a16_gemv_prefetch_l2.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, sz, vp, u32,
                                           ctypes.POINTER(L2Range), i32, vp]
    lib.w4a16_gemv_static_scratch.restype = i32
    lib.w4a16_gemv_static_scratch.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, u32, vp]
    lib.w4a16_gemv_workspace_bytes.restype = sz
    lib.w4a16_gemv_workspace_bytes.argtypes = [i32, i32, i32]
    lib.w4a16_gemv_workspace_bytes_flags.restype = sz
    lib.w4a16_gemv_workspace_bytes_flags.argtypes = [i32, i32, i32, ctypes.c_uint]
    lib.w4a16_gemv_id.restype = i32
    lib.w4a16_gemv_id.argtypes = [vp, vp, sz, vp, sz, i32, vp, i32, vp, i32, i32, i32, vp, u32, vp]
    lib.w4a16_gemv_id_scaled.restype = i32
    lib.w4a16_gemv_id_scaled.argtypes = [vp, vp, sz, vp, sz, i32, vp, i32, vp, i32, i32, i32,
                                         vp, i32, vp, vp, vp, vp, u32, vp]
    lib.w4_embed_gather.restype = i32
    lib.w4_embed_gather.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, u32, vp]
    lib.w4_pack.restype = i32
    lib.w4_pack.argtypes = [vp, vp, i32, i32, vp, vp]
    lib.w4_quantize.restype = i32
    lib.w4_quantize.argtypes = [vp, vp, vp, i32, i32, vp]
    lib.w4_slot_pool_create.restype = i32
    lib.w4_slot_pool_create.argtypes = [ctypes.POINTER(vp), i32, i32]
    lib.w4_slot_pool_destroy.restype = None
    lib.w4_slot_pool_destroy.argtypes = [vp]
    lib.w4_slot_pool_remap.restype = i32
    lib.w4_slot_pool_remap.argtypes = [vp, i32p, i32, i32p, i32p, i32p, ctypes.POINTER(i32)]
    lib.w4_slot_pool_stage.restype = i32
    lib.w4_slot_pool_stage.argtypes = [vp, i32p, i32, vp, vp, sz, sz, vp, vp, sz, sz, vp, vp,
                                       i32p, ctypes.POINTER(i32), vp]
    lib.w4_slot_pool_stats.restype = None
    lib.w4_slot_pool_stats.argtypes = [vp] + [ctypes.POINTER(ctypes.c_longlong)] * 3
    lib.w4_dev_pool_state_bytes.restype = sz
    lib.w4_dev_pool_state_bytes.argtypes = [i32, i32]
    lib.w4_dev_pool_init.restype = i32
    lib.w4_dev_pool_init.argtypes = [vp, i32, i32, vp]
    lib.w4_dev_pool_stage.restype = i32
    lib.w4_dev_pool_stage.argtypes = [vp, i32, i32, vp, i32, vp, vp, sz, sz, vp, vp, sz, sz, vp,
                                      vp, vp, u32, vp]
    lib.w4_dev_pool_stats.restype = i32
    lib.w4_dev_pool_stats.argtypes = [vp, i32, i32] + [ctypes.POINTER(ctypes.c_longlong)] * 3
    lib.w4a16_gemv_plan.restype = i32
    lib.w4a16_gemv_plan.argtypes = [i32, i32, i32, ctypes.POINTER(PlanInfo)]
    lib.w4a16_gemv_plan_flags.restype = i32
    lib.w4a16_gemv_plan_flags.argtypes = [i32, i32, i32, u32, ctypes.POINTER(PlanInfo)]
    lib.w4a16_gemv_id_plan.restype = i32
    lib.w4a16_gemv_id_plan.argtypes = [i32, i32, i32, i32, ctypes.POINTER(PlanInfo)]
    lib.w4a16_gemv_chain.restype = i32
    lib.w4a16_gemv_chain.argtypes = [ctypes.POINTER(GemvTask), i32, vp, sz, vp, u32, vp]
    lib.w4a16_gemv_chain_workspace_bytes.restype = sz
    lib.w4a16_gemv_chain_workspace_bytes.argtypes = [ctypes.POINTER(GemvTask), i32]
    lib.w4a16_gemv_chain_plan.restype = i32
    lib.w4a16_gemv_chain_plan.argtypes = [ctypes.POINTER(GemvTask), i32,
                                          ctypes.POINTER(ChainPlanInfo)]
    lib.w4a16_gemv_chain_task_plan.restype = i32
    lib.w4a16_gemv_chain_task_plan.argtypes = [ctypes.POINTER(GemvTask), i32, i32,
                                               ctypes.POINTER(ChainTaskInfo)]
    _lib = lib
    return lib


def _check(code: int, what: str):
    if code != 0:
        if code in (5, 10):
            what = f"{what} ({load().w4_last_cuda_error().decode()})"
        raise W4Error(code, what)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _as_words(qw: torch.Tensor) -> torch.Tensor:
    if qw.dtype not in (torch.int32, torch.uint32):
        raise ValueError("qw must hold 32-bit words (int32 or uint32)")
    return qw


# ------------------------------------------------------------------ calls
def workspace_bytes(M: int, N: int, K: int, path: str = None) -> int:
    """Zero-filled scratch a gemv call of this shape (and path choice) needs."""
    if path is None:
        return int(load().w4a16_gemv_workspace_bytes(M, N, K))
    return int(load().w4a16_gemv_workspace_bytes_flags(M, N, K, _PATH_FLAGS[path]))


def plan(M: int, N: int, K: int, path: str = None) -> dict:
    """Launch plan of a w4a16_gemv call (path: None, "cuda" or "tensor")."""
    info = PlanInfo()
    _check(load().w4a16_gemv_plan_flags(M, N, K, _PATH_FLAGS[path], ctypes.byref(info)),
           "w4a16_gemv_plan_flags")
    return {n: getattr(info, n) for n, _ in PlanInfo._fields_}


def id_plan(n_ids: int, x_rows: int, N: int, K: int) -> dict:
    """Launch plan of a w4a16_gemv_id call."""
    info = PlanInfo()
    _check(load().w4a16_gemv_id_plan(n_ids, x_rows, N, K, ctypes.byref(info)),
           "w4a16_gemv_id_plan")
    return {n: getattr(info, n) for n, _ in PlanInfo._fields_}


def l2_ranges(ranges):
    """A ctypes array of w4_l2_range from (tensor, bytes) or (address, bytes)
    pairs (bytes None: the whole tensor)."""
    arr = (L2Range * max(1, len(ranges)))()
    for i, (t, nbytes) in enumerate(ranges):
        if isinstance(t, torch.Tensor):
            _need(t, t.dtype, "prefetch range")
            full = t.numel() * t.element_size()
            nbytes = full if nbytes is None else min(int(nbytes), full)
            arr[i] = L2Range(t.data_ptr(), nbytes)
        else:
            arr[i] = L2Range(int(t), int(nbytes))
    return arr


def gemv(qw: torch.Tensor, st: torch.Tensor, x: torch.Tensor, y: torch.Tensor = None,
         workspace: torch.Tensor = None, status: torch.Tensor = None, pdl: bool = False,
         stream=None, path: str = None, silu_mul: bool = False, l2_next=None) -> torch.Tensor:
    """y[M, N] = x[M, K] @ W^T with W from (qw [N, K/8], st [N, K/32]).

    path: None (the library's choice), "cuda" (CUDA cores) or "tensor"
    (tcgen05 tensor cores; K a multiple of 256).
    silu_mul: x is [M, 2K] (gate then up) and the product takes
    silu(gate) * up, formed while the activations are staged.
    l2_next: up to 4 (tensor or address, bytes) ranges, normally the next
    call's codes and steps, brought into L2 once this call has requested its
    own weights (w4a16_gemv_prefetch_l2)."""
    qw = _as_words(qw)
    _need(qw, qw.dtype, "qw")
    _need(st, torch.bfloat16, "st")
    _need(x, torch.bfloat16, "x")
    x2 = x if x.dim() == 2 else x.view(1, -1)
    M, K = x2.shape
    if silu_mul:
        if K % 2:
            raise ValueError("silu_mul needs x rows of [gate | up]")
        K //= 2
    N = qw.shape[0]
    if qw.shape != (N, K // 8) or st.shape != (N, K // 32):
        raise ValueError("qw/st shapes do not match x")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(y, torch.bfloat16, "y")
    # workspace: zero-filled, workspace_bytes(M, N, K, path) large.  The
    # library refuses a call whose K split needs it (W4_ERR_WORKSPACE); a
    # tensor-core call that only uses it for balanced runs runs without it.
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    flags = (W4_FLAG_PDL if pdl else 0) | _PATH_FLAGS[path] | (W4_FLAG_SILU_MUL if silu_mul else 0)
    if l2_next:
        if len(l2_next) > W4_MAX_L2_RANGES:
            raise ValueError(f"at most {W4_MAX_L2_RANGES} prefetch ranges")
        rs = l2_next if isinstance(l2_next, ctypes.Array) else l2_ranges(l2_next)
        _check(load().w4a16_gemv_prefetch_l2(_ptr(y), _ptr(qw), _ptr(st), _ptr(x2), M, N, K,
                                             _ptr(workspace), ws_bytes, _ptr(status), flags, rs,
                                             len(rs), _stream(stream)),
               "w4a16_gemv_prefetch_l2")
        return y
    _check(load().w4a16_gemv(_ptr(y), _ptr(qw), _ptr(st), _ptr(x2), M, N, K, _ptr(workspace),
                             ws_bytes, _ptr(status), flags, _stream(stream)),
           "w4a16_gemv")
    return y


def gemv_id(qw_base: torch.Tensor, st_base: torch.Tensor, ids: torch.Tensor, x: torch.Tensor,
            N: int, K: int, num_experts: int, qw_stride_bytes: int, st_stride_bytes: int,
            y: torch.Tensor = None, status: torch.Tensor = None, pdl: bool = False,
            stream=None, ids_final: bool = False) -> torch.Tensor:
    """y[i] = W_{ids[i]} @ x[i or 0]; experts at base + id * stride (bytes)."""
    _need(ids, torch.int32, "ids")
    _need(x, torch.bfloat16, "x")
    if not (qw_base.is_cuda and st_base.is_cuda):
        raise ValueError("bases must be CUDA tensors")
    x2 = x if x.dim() == 2 else x.view(1, -1)
    n_ids = ids.numel()
    if y is None:
        y = torch.empty((n_ids, N), dtype=torch.bfloat16, device=x.device)
    _need(y, torch.bfloat16, "y")
    _check(load().w4a16_gemv_id(_ptr(y), _ptr(qw_base), qw_stride_bytes, _ptr(st_base),
                                st_stride_bytes, num_experts, _ptr(ids), n_ids, _ptr(x2),
                                x2.shape[0], N, K, _ptr(status), _id_flags(pdl, ids_final),
                                _stream(stream)), "w4a16_gemv_id")
    return y


def bind_gemv_id(qw_base: torch.Tensor, st_base: torch.Tensor, ids: torch.Tensor,
                 x: torch.Tensor, N: int, K: int, num_experts: int, qw_stride_bytes: int,
                 st_stride_bytes: int, y: torch.Tensor, status: torch.Tensor = None):
    """w4a16_gemv_id with its arguments marshalled once, for decode loops.

    Returns call(pdl=False, stream=None), which enqueues the same routed
    product again (reading whatever the tensors hold at that time; they must
    stay allocated and in place).
    """
    _need(ids, torch.int32, "ids")
    _need(x, torch.bfloat16, "x")
    _need(y, torch.bfloat16, "y")
    if not (qw_base.is_cuda and st_base.is_cuda):
        raise ValueError("bases must be CUDA tensors")
    x2 = x if x.dim() == 2 else x.view(1, -1)
    fn = load().w4a16_gemv_id
    args = (_ptr(y), _ptr(qw_base), qw_stride_bytes, _ptr(st_base), st_stride_bytes, num_experts,
            _ptr(ids), ids.numel(), _ptr(x2), x2.shape[0], N, K, _ptr(status))

    def call(pdl: bool = False, stream=None, ids_final: bool = False):
        _check(fn(*args, _id_flags(pdl, ids_final), _stream(stream)), "w4a16_gemv_id")

    call.tensors = (qw_base, st_base, ids, x2, y, status)   # keep them alive
    return call


def _scaled_args(y, qw_base, qw_stride_bytes, st_base, st_stride_bytes, num_slots, ids, x, N, K,
                 expert_ids, num_experts, slot_expert, scale, bias, status):
    _need(ids, torch.int32, "ids")
    _need(expert_ids, torch.int32, "expert_ids")
    _need(x, torch.bfloat16, "x")
    _need(y, torch.bfloat16, "y")
    if expert_ids.numel() != ids.numel():
        raise ValueError("expert_ids must have one entry per id")
    if slot_expert is not None:
        _need(slot_expert, torch.int32, "slot_expert")
    for name, t in (("scale", scale), ("bias", bias)):
        if t is not None:
            _need(t, torch.bfloat16, name)
            if t.numel() != num_experts * N:
                raise ValueError(f"{name} must be [num_experts][N]")
    if not (qw_base.is_cuda and st_base.is_cuda):
        raise ValueError("bases must be CUDA tensors")
    x2 = x if x.dim() == 2 else x.view(1, -1)
    return x2, (_ptr(y), _ptr(qw_base), qw_stride_bytes, _ptr(st_base), st_stride_bytes,
                num_slots, _ptr(ids), ids.numel(), _ptr(x2), x2.shape[0], N, K, _ptr(expert_ids),
                num_experts, _ptr(slot_expert), _ptr(scale), _ptr(bias), _ptr(status))


def gemv_id_scaled(qw_base: torch.Tensor, st_base: torch.Tensor, ids: torch.Tensor,
                   x: torch.Tensor, N: int, K: int, num_slots: int, qw_stride_bytes: int,
                   st_stride_bytes: int, expert_ids: torch.Tensor, num_experts: int,
                   slot_expert: torch.Tensor = None, scale: torch.Tensor = None,
                   bias: torch.Tensor = None, y: torch.Tensor = None,
                   status: torch.Tensor = None, pdl: bool = False, stream=None,
                   ids_final: bool = False) -> torch.Tensor:
    """y[i] = bf16(fma(W_{ids[i]} @ x[i or 0], scale[e], bias[e])), e = expert_ids[i]:
    weights through slot (or expert) ids, per-expert vectors through real ids."""
    if y is None:
        y = torch.empty((ids.numel(), N), dtype=torch.bfloat16, device=x.device)
    _, args = _scaled_args(y, qw_base, qw_stride_bytes, st_base, st_stride_bytes, num_slots, ids,
                           x, N, K, expert_ids, num_experts, slot_expert, scale, bias, status)
    _check(load().w4a16_gemv_id_scaled(*args, _id_flags(pdl, ids_final), _stream(stream)),
           "w4a16_gemv_id_scaled")
    return y


def bind_gemv_id_scaled(qw_base, st_base, ids, x, N, K, num_slots, qw_stride_bytes,
                        st_stride_bytes, expert_ids, num_experts, y, slot_expert=None,
                        scale=None, bias=None, status=None):
    """w4a16_gemv_id_scaled with its arguments marshalled once: returns
    call(pdl=False, stream=None)."""
    x2, args = _scaled_args(y, qw_base, qw_stride_bytes, st_base, st_stride_bytes, num_slots,
                            ids, x, N, K, expert_ids, num_experts, slot_expert, scale, bias,
                            status)
    fn = load().w4a16_gemv_id_scaled

    def call(pdl: bool = False, stream=None, ids_final: bool = False):
        _check(fn(*args, _id_flags(pdl, ids_final), _stream(stream)), "w4a16_gemv_id_scaled")

    call.tensors = (qw_base, st_base, ids, x2, y, expert_ids, slot_expert, scale, bias, status)
    return call


def embed_gather(qw: torch.Tensor, st: torch.Tensor, ids: torch.Tensor, out: torch.Tensor = None,
                 status: torch.Tensor = None, pdl: bool = False, stream=None) -> torch.Tensor:
    qw = _as_words(qw)
    _need(qw, qw.dtype, "qw")
    _need(st, torch.bfloat16, "st")
    _need(ids, torch.int32, "ids")
    V, K = qw.shape[0], qw.shape[1] * 8
    T = ids.numel()
    if out is None:
        out = torch.empty((T, K), dtype=torch.bfloat16, device=qw.device)
    _need(out, torch.bfloat16, "out")
    _check(load().w4_embed_gather(_ptr(out), _ptr(qw), _ptr(st), _ptr(ids), T, V, K, _ptr(status),
                                  W4_FLAG_PDL if pdl else 0, _stream(stream)), "w4_embed_gather")
    return out


def pack(codes: torch.Tensor, qw: torch.Tensor = None, status: torch.Tensor = None,
         stream=None) -> torch.Tensor:
    _need(codes, torch.uint8, "codes")
    N, K = codes.shape
    if qw is None:
        qw = torch.empty((N, K // 8), dtype=torch.int32, device=codes.device)
    _check(load().w4_pack(_ptr(qw), _ptr(codes), N, K, _ptr(status), _stream(stream)), "w4_pack")
    return qw


def quantize(w: torch.Tensor, stream=None):
    _need(w, torch.float32, "w")
    N, K = w.shape
    qw = torch.empty((N, K // 8), dtype=torch.int32, device=w.device)
    st = torch.empty((N, K // 32), dtype=torch.bfloat16, device=w.device)
    _check(load().w4_quantize(_ptr(qw), _ptr(st), _ptr(w), N, K, _stream(stream)), "w4_quantize")
    return qw, st


class DevSlotPool:
    """Device-side LFU expert-slot pool: state in a device buffer, remap and
    fills enqueued on a stream (graph-capturable)."""

    def __init__(self, num_experts: int, num_slots: int, device="cuda", stream=None):
        self._lib = load()
        n = self._lib.w4_dev_pool_state_bytes(num_experts, num_slots)
        if n == 0:
            raise W4Error(3, "w4_dev_pool_state_bytes")
        self.state = torch.empty(n, dtype=torch.uint8, device=device)
        self.num_experts, self.num_slots = num_experts, num_slots
        self.reset(stream)

    def reset(self, stream=None):
        """Every slot free, every count 0 (enqueued on `stream`)."""
        _check(self._lib.w4_dev_pool_init(_ptr(self.state), self.num_experts, self.num_slots,
                                          _stream(stream)), "w4_dev_pool_init")

    def bind_stage(self, ids_dev: torch.Tensor, pool_qw, full_qw, qw_stride, qw_bytes, pool_st,
                   full_st, st_stride, st_bytes, slot_ids_dev: torch.Tensor, slot_expert=None,
                   status=None):
        """Returns call(pdl=False, stream=None) that enqueues the remap of the
        ids then held by ids_dev (device int32 [k]) and the fills."""
        _need(ids_dev, torch.int32, "ids_dev")
        _need(slot_ids_dev, torch.int32, "slot_ids_dev")
        fn = self._lib.w4_dev_pool_stage
        args = (_ptr(self.state), self.num_experts, self.num_slots, _ptr(ids_dev), ids_dev.numel(),
                _ptr(pool_qw), _ptr(full_qw), qw_stride, qw_bytes, _ptr(pool_st), _ptr(full_st),
                st_stride, st_bytes, _ptr(slot_ids_dev), _ptr(slot_expert), _ptr(status))

        def call(pdl: bool = False, stream=None):
            _check(fn(*args, W4_FLAG_PDL if pdl else 0, _stream(stream)), "w4_dev_pool_stage")

        call.tensors = (self.state, ids_dev, pool_qw, full_qw, pool_st, full_st, slot_ids_dev,
                        slot_expert, status)
        return call

    def stats(self):
        r, h, m = ctypes.c_longlong(), ctypes.c_longlong(), ctypes.c_longlong()
        _check(self._lib.w4_dev_pool_stats(_ptr(self.state), self.num_experts, self.num_slots,
                                           ctypes.byref(r), ctypes.byref(h), ctypes.byref(m)),
               "w4_dev_pool_stats")
        return {"requests": r.value, "hits": h.value, "misses": m.value}


class SlotPool:
    """Host LFU expert-slot pool (C++ in the library)."""

    def __init__(self, num_experts: int, num_slots: int):
        self._lib = load()
        h = ctypes.c_void_p()
        _check(self._lib.w4_slot_pool_create(ctypes.byref(h), num_experts, num_slots),
               "w4_slot_pool_create")
        self._h = h
        self.num_experts, self.num_slots = num_experts, num_slots

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self._lib.w4_slot_pool_destroy(h)
            self._h = None

    def remap(self, ids):
        ids = [int(v) for v in ids]
        k = len(ids)
        arr = (ctypes.c_int32 * k)(*ids)
        slots = (ctypes.c_int32 * k)()
        me = (ctypes.c_int32 * k)()
        ms = (ctypes.c_int32 * k)()
        nm = ctypes.c_int()
        _check(self._lib.w4_slot_pool_remap(self._h, arr, k, slots, me, ms, ctypes.byref(nm)),
               "w4_slot_pool_remap")
        return list(slots), [(me[i], ms[i]) for i in range(nm.value)]

    def stage(self, ids, pool_qw, full_qw, qw_stride, qw_bytes, pool_st, full_st, st_stride,
              st_bytes, slot_ids_dev: torch.Tensor, stream=None, slot_expert=None):
        """Remap, copy missed experts into the pool and write slot ids (and, when
        given, the device slot table), all on `stream`.  full_qw / full_st may
        be CUDA tensors or page-locked CPU tensors."""
        ids = [int(v) for v in ids]
        k = len(ids)
        arr = (ctypes.c_int32 * k)(*ids)
        slots = (ctypes.c_int32 * k)()
        nm = ctypes.c_int()
        _check(self._lib.w4_slot_pool_stage(self._h, arr, k, _ptr(pool_qw), _ptr(full_qw),
                                            qw_stride, qw_bytes, _ptr(pool_st), _ptr(full_st),
                                            st_stride, st_bytes, _ptr(slot_ids_dev),
                                            _ptr(slot_expert), slots, ctypes.byref(nm),
                                            _stream(stream)),
               "w4_slot_pool_stage")
        return list(slots), nm.value

    def bind_stage(self, k: int, pool_qw, full_qw, qw_stride, qw_bytes, pool_st, full_st,
                   st_stride, st_bytes, slot_ids_dev: torch.Tensor, slot_expert=None):
        """stage() with the buffers marshalled once: returns call(ids, stream=None)
        for requests of k ids (any int sequence), which returns the misses."""
        arr = (ctypes.c_int32 * k)()
        slots = (ctypes.c_int32 * k)()
        nm = ctypes.c_int()
        fixed = (_ptr(pool_qw), _ptr(full_qw), qw_stride, qw_bytes, _ptr(pool_st), _ptr(full_st),
                 st_stride, st_bytes, _ptr(slot_ids_dev), _ptr(slot_expert), slots,
                 ctypes.byref(nm))
        fn, h = self._lib.w4_slot_pool_stage, self._h

        def call(ids, stream=None) -> int:
            if len(ids) != k:
                raise ValueError(f"expected {k} ids")
            for i, v in enumerate(ids):
                arr[i] = int(v)
            _check(fn(h, arr, k, *fixed, _stream(stream)), "w4_slot_pool_stage")
            return nm.value

        call.tensors = (pool_qw, full_qw, pool_st, full_st, slot_ids_dev, slot_expert)
        return call

    def stats(self):
        r, h, m = ctypes.c_longlong(), ctypes.c_longlong(), ctypes.c_longlong()
        self._lib.w4_slot_pool_stats(self._h, ctypes.byref(r), ctypes.byref(h), ctypes.byref(m))
        return {"requests": r.value, "hits": h.value, "misses": m.value}


# ------------------------------------------------------------------ chains
def gemv_task(qw: torch.Tensor, st: torch.Tensor, x: torch.Tensor, y: torch.Tensor, dep: int = -1,
              silu_mul: bool = False) -> dict:
    """A dense task of a chain: y[N] = W x (x [K], or [2K] = [gate | up] with silu_mul)."""
    qw = _as_words(qw)
    for t, dt, name in ((qw, qw.dtype, "qw"), (st, torch.bfloat16, "st"),
                        (x, torch.bfloat16, "x"), (y, torch.bfloat16, "y")):
        _need(t, dt, name)
    N, K = qw.shape[0], qw.shape[-1] * 8
    if st.shape[0] != N or st.shape[-1] != K // 32 or y.numel() != N:
        raise ValueError("qw, st and y disagree on N or K")
    if x.numel() != K * (2 if silu_mul else 1):
        raise ValueError("x must hold one activation row")
    return {"y": y, "qw": qw, "st": st, "x": x, "ids": None, "qw_stride": 0, "st_stride": 0,
            "num_experts": 0, "n_ids": 1, "x_rows": 1, "N": N, "K": K, "dep": dep,
            "flags": W4_TASK_SILU_MUL if silu_mul else 0}


def gemv_id_task(qw_base: torch.Tensor, st_base: torch.Tensor, ids: torch.Tensor,
                 x: torch.Tensor, y: torch.Tensor, N: int, K: int, num_experts: int,
                 qw_stride_bytes: int, st_stride_bytes: int, dep: int = -1,
                 silu_mul: bool = False) -> dict:
    """A routed task of a chain: y[i] = W_{ids[i]} x_i (x_i: row i when x has
    n_ids rows, else row 0; [gate | up] rows of 2K with silu_mul)."""
    _need(ids, torch.int32, "ids")
    _need(x, torch.bfloat16, "x")
    _need(y, torch.bfloat16, "y")
    n_ids = ids.numel()
    row = K * (2 if silu_mul else 1)
    if x.numel() % row or x.numel() // row not in (1, n_ids):
        raise ValueError("x must hold 1 or n_ids activation rows")
    if y.numel() != n_ids * N:
        raise ValueError("y must be [n_ids, N]")
    return {"y": y, "qw": qw_base, "st": st_base, "x": x, "ids": ids,
            "qw_stride": qw_stride_bytes, "st_stride": st_stride_bytes,
            "num_experts": num_experts, "n_ids": n_ids, "x_rows": x.numel() // row, "N": N,
            "K": K, "dep": dep, "flags": W4_TASK_SILU_MUL if silu_mul else 0}


def _task_array(tasks):
    arr = (GemvTask * len(tasks))()
    for i, t in enumerate(tasks):
        g = arr[i]
        for name in ("y", "qw", "st", "x", "ids"):
            setattr(g, name, None if t[name] is None else t[name].data_ptr())
        for name in ("qw_stride", "st_stride", "num_experts", "n_ids", "x_rows", "N", "K", "dep",
                     "flags"):
            setattr(g, name, int(t[name]))
    return arr


def chain_workspace_bytes(tasks) -> int:
    """Bytes of the zero-initialised workspace a chain of these tasks needs."""
    return int(load().w4a16_gemv_chain_workspace_bytes(_task_array(tasks), len(tasks)))


def chain_plan(tasks) -> dict:
    arr = _task_array(tasks)
    info = ChainPlanInfo()
    _check(load().w4a16_gemv_chain_plan(arr, len(tasks), ctypes.byref(info)),
           "w4a16_gemv_chain_plan")
    return {n: getattr(info, n) for n, _ in ChainPlanInfo._fields_}


def chain_task_plan(tasks, task: int) -> dict:
    arr = _task_array(tasks)
    info = ChainTaskInfo()
    _check(load().w4a16_gemv_chain_task_plan(arr, len(tasks), task, ctypes.byref(info)),
           "w4a16_gemv_chain_task_plan", "w4a16_gemv_id_plan")
    return {n: getattr(info, n) for n, _ in ChainTaskInfo._fields_}


def bind_gemv_chain(tasks, workspace: torch.Tensor, status: torch.Tensor = None):
    """w4a16_gemv_chain with the task list marshalled once: returns
    call(pdl=False, stream=None).  `workspace` (uint8, zeroed once) must hold
    chain_workspace_bytes(tasks) bytes."""
    _need(workspace, torch.uint8, "workspace")
    arr = _task_array(tasks)
    n = len(tasks)
    fn = load().w4a16_gemv_chain
    ws_ptr, ws_bytes = _ptr(workspace), workspace.numel()

    def call(pdl: bool = False, stream=None):
        _check(fn(arr, n, ws_ptr, ws_bytes, _ptr(status), W4_FLAG_PDL if pdl else 0,
                  _stream(stream)), "w4a16_gemv_chain")

    call.tensors = (tasks, workspace, status)   # keep the buffers alive with the binding
    return call


def gemv_chain(tasks, workspace: torch.Tensor, status: torch.Tensor = None, pdl: bool = False,
               stream=None):
    """Run the tasks (dicts from gemv_task / gemv_id_task) as one launch."""
    bind_gemv_chain(tasks, workspace, status)(pdl=pdl, stream=stream)
