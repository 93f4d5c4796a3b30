"""GB300 ring attention -- forward, backward and the context-parallel variants:
the Python binding of libra.so (include/ra.h).

The functions keep the C names (``ra_plan``, ``ra_plan_tile_counts``, ``ra_fwd``,
``ra_fwd_static``, ``ra_fwd_static_status``, ``ra_merge_partials``, ``ra_layout_perm``, ``ra_layout_index``,
``ra_fwd_step``, ``ra_ring_rotate``, ``ra_ring_fwd``, ``ra_bwd``,
``ra_bwd_scratch_size``, ``ra_allgather_kv``, ``ra_fwd_gathered``,
``ra_ulysses_a2a``, ``ra_sync_status``, ``ra_wait_selftest``, ``ra_last_error``).
This module only marshals arguments: PyTorch supplies device memory and the
current stream, every step of the computation runs in the library's CUDA
kernels, and there is no fallback -- if libra.so is missing or cannot be loaded,
every call raises.  Because the library sees only pointers, every tensor a caller
passes (outputs and scratch included) is checked here for its exact shape, dtype,
contiguity and device before anything is launched.

Tensors are ``[B, H, S, d]`` contiguous with S in layout order (shard p owns rows
[p*S/N, (p+1)*S/N)); ``ra_layout_perm`` moves natural order <-> layout order.

With RA_LIBRARY_VARIANT=debug in the environment the binding loads libra_debug.so
instead: the same library with the kernels' bounds checks compiled in, which
``ra_sync_status`` reports as RaError(RA_ERR_BOUNDS).
"""

import ctypes
import os

import numpy as np

__all__ = [
    "RaError", "Plan", "LAYOUTS",
    "ra_plan", "ra_plan_destroy", "ra_plan_tile_counts", "ra_fwd", "ra_merge_partials",
    "ra_layout_perm", "ra_layout_index", "ra_sync_status", "ra_last_error", "ra_fwd_static",
    "ra_fwd_static_status", "ra_fwd_step", "ra_ring_rotate", "ra_ring_fwd", "ra_bwd", "ra_bwd_scratch_size",
    "ra_allgather_kv", "ra_fwd_gathered", "ra_ulysses_a2a", "ra_wait_selftest",
    "library_path", "load_library", "EXPORTED",
]

LAYOUTS = {"contiguous": 0, "striped": 1, "zigzag": 2}
DTYPES = {"f32": 0, "bf16": 1}
_STATUS = {0: "RA_OK", 1: "RA_ERR_INVALID_ARG", 2: "RA_ERR_UNSUPPORTED", 3: "RA_ERR_CUDA",
           4: "RA_ERR_TIMEOUT", 5: "RA_ERR_NO_DEVICE", 6: "RA_ERR_BOUNDS"}
EXPORTED = ("ra_plan", "ra_plan_destroy", "ra_plan_tile_counts", "ra_fwd", "ra_merge_partials",
            "ra_layout_perm", "ra_layout_index", "ra_sync_status", "ra_last_error", "ra_fwd_static",
            "ra_fwd_static_status", "ra_fwd_step", "ra_ring_rotate", "ra_ring_fwd", "ra_bwd", "ra_bwd_scratch_size",
            "ra_allgather_kv", "ra_fwd_gathered", "ra_ulysses_a2a", "ra_wait_selftest")

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


class RaError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        self.name = _STATUS.get(status, str(status))
        super().__init__(f"{self.name}: {message}")


class _Problem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seq", ctypes.c_int64), ("heads_q", ctypes.c_int32),
                ("heads_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("n_shards", ctypes.c_int32),
                ("layout", ctypes.c_int32), ("causal", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("scale", ctypes.c_float)]


def library_path():
    """libra.so, or with RA_LIBRARY_VARIANT=debug in the environment libra_debug.so: the same
    library with the kernels' bounds checks compiled in (built by build.build_all())."""
    name = "libra_debug.so" if os.environ.get("RA_LIBRARY_VARIANT") == "debug" else "libra.so"
    return os.path.join(_HERE, name)


def load_library():
    """Load libra.so (built in-tree by ``build.build()``); raises if it is absent."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run context_ring_attention_gb300.build.build_all()")
    lib = ctypes.CDLL(path)
    P, I32, I64, VP = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    sig = {
        "ra_plan": ([ctypes.POINTER(_Problem), ctypes.POINTER(P)], I32),
        "ra_plan_destroy": ([P], I32),
        "ra_plan_tile_counts": ([P, VP, VP, VP], I32),
        "ra_fwd": ([P, VP, VP, VP, VP, VP, VP, VP, VP], I32),
        "ra_merge_partials": ([I32, I64, I32, VP, VP, VP, I32, VP, VP], I32),
        "ra_layout_perm": ([I32, I64, I32, I32, I64, I32, VP, VP, VP], I32),
        "ra_layout_index": ([I32, I64, I32, VP], I32),
        "ra_sync_status": ([P, VP], I32),
        "ra_last_error": ([], ctypes.c_char_p),
        "ra_fwd_static": ([ctypes.POINTER(_Problem), VP, VP, VP, VP, VP, VP], I32),
        "ra_fwd_static_status": ([VP], I32),
        "ra_fwd_step": ([P, I32, VP, VP, VP, VP, VP, VP], I32),
        "ra_ring_rotate": ([P, VP, VP, VP, VP, VP], I32),
        "ra_ring_fwd": ([P, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP], I32),
        "ra_bwd": ([P, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP], I32),
        "ra_bwd_scratch_size": ([P, VP], I32),
        "ra_allgather_kv": ([P, VP, VP, VP, VP, VP], I32),
        "ra_fwd_gathered": ([P, VP, VP, VP, VP, VP, VP], I32),
        "ra_ulysses_a2a": ([I32, I32, I64, I32, I64, I32, I32, VP, VP, VP], I32),
        "ra_wait_selftest": ([VP], I32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _LIB = lib
    return lib


def ra_last_error():
    return load_library().ra_last_error().decode()


def _check(status):
    if status != 0:
        raise RaError(status, ra_last_error())


def _layout(layout):
    return LAYOUTS[layout] if isinstance(layout, str) else int(layout)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    cur = torch.cuda.current_device()
    if stream.device.index != cur:
        raise ValueError(f"the stream belongs to {stream.device}; the library launches on the current device "
                         f"cuda:{cur}")
    return ctypes.c_void_p(stream.cuda_stream)


def _on_current_device(name, t):
    """The kernels run on the current CUDA device: every buffer must live there."""
    import torch
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    cur = torch.cuda.current_device()
    if t.device.index != cur:
        raise ValueError(f"{name} is on {t.device}, but the current device is cuda:{cur} "
                         f"(make its device current, e.g. with torch.cuda.device)")


class Plan:
    """Owns an ``ra_plan_t``; the problem it was built for is ``self.problem``."""

    def __init__(self, handle, problem):
        self._h = handle
        self.problem = problem

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h:
            load_library().ra_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def ra_plan(batch, seq, heads_q, heads_kv, head_dim, n_shards, layout="contiguous",
            causal=False, dtype="bf16", scale=0.0):
    """Validate a problem and build its ring schedule (see include/ra.h)."""
    lib = load_library()
    dt = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    prob = _Problem(int(batch), int(seq), int(heads_q), int(heads_kv), int(head_dim), int(n_shards),
                    _layout(layout), int(bool(causal)), dt, float(scale or 0.0))
    h = ctypes.c_void_p()
    _check(lib.ra_plan(ctypes.byref(prob), ctypes.byref(h)))
    info = dict(batch=int(batch), seq=int(seq), heads_q=int(heads_q), heads_kv=int(heads_kv),
                head_dim=int(head_dim), n_shards=int(n_shards), layout=_layout(layout),
                causal=bool(causal), dtype=dt, scale=float(scale or 0.0))
    return Plan(h, info)


def ra_plan_destroy(plan):
    plan.close()


def ra_plan_tile_counts(plan):
    """Per-shard (FULL, PARTIAL, SKIP) tile counts of one (batch, query head)."""
    n = plan.problem["n_shards"]
    full, part, skip = (np.zeros(n, np.int64) for _ in range(3))
    _check(load_library().ra_plan_tile_counts(plan.handle, full.ctypes.data, part.ctypes.data,
                                              skip.ctypes.data))
    return full, part, skip


def _check_qkv(plan, **tensors):
    """Shape/dtype/contiguity of q ([B, Hq, S, d]) and K/V-like ([B, Hkv, S, d]) arguments."""
    import torch
    pb = plan.problem
    B, S, d = pb["batch"], pb["seq"], pb["head_dim"]
    dt = torch.bfloat16 if pb["dtype"] == 1 else torch.float32
    for name, t in tensors.items():
        heads = pb["heads_q"] if name == "q" else pb["heads_kv"]
        if tuple(t.shape) != (B, heads, S, d) or t.dtype != dt or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor of shape {(B, heads, S, d)}")
        _on_current_device(name, t)


def _need(name, t, shape, dtype, device):
    """``t`` must be a contiguous tensor of exactly this shape and dtype on ``device``:
    the library sees only its pointer, so a smaller buffer would be overrun."""
    import torch
    if (not isinstance(t, torch.Tensor) or tuple(t.shape) != tuple(int(x) for x in shape) or t.dtype != dtype
            or not t.is_contiguous() or t.device != device):
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} on {device}")
    _on_current_device(name, t)


def _same_device(device, **tensors):
    for name, t in tensors.items():
        if t.device != device:
            raise ValueError(f"{name} is on {t.device}, the other tensors on {device}")


def ra_fwd(plan, q, k, v, o=None, lse=None, partials=False, o_parts=None, lse_parts=None,
           stream=None):
    """Ring-attention forward.  Fused: returns (O, LSE).  partials=True: (O_parts, LSE_parts)."""
    import torch
    pb = plan.problem
    B, Hq, S, d, N = pb["batch"], pb["heads_q"], pb["seq"], pb["head_dim"], pb["n_shards"]
    _check_qkv(plan, q=q, k=k, v=v)
    _same_device(q.device, k=k, v=v)
    lib = load_library()
    if partials:
        if o_parts is None:
            o_parts = torch.empty((N, B, Hq, S, d), dtype=torch.float32, device=q.device)
        if lse_parts is None:
            lse_parts = torch.empty((N, B, Hq, S), dtype=torch.float32, device=q.device)
        _need("o_parts", o_parts, (N, B, Hq, S, d), torch.float32, q.device)
        _need("lse_parts", lse_parts, (N, B, Hq, S), torch.float32, q.device)
        _check(lib.ra_fwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), None, None, _ptr(o_parts),
                          _ptr(lse_parts), _stream(stream)))
        return o_parts, lse_parts
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    _need("o", o, q.shape, q.dtype, q.device)
    _need("lse", lse, (B, Hq, S), torch.float32, q.device)
    _check(lib.ra_fwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), None, None,
                      _stream(stream)))
    return o, lse


def ra_merge_partials(o_parts, lse_parts, out_dtype=None, o=None, lse=None, stream=None):
    """Merge [n, ..., d] partial outputs with their [n, ...] LSEs -> (O, LSE)."""
    import torch
    n, d = o_parts.shape[0], o_parts.shape[-1]
    rows = lse_parts[0].numel()
    if o_parts.dtype != torch.float32 or lse_parts.dtype != torch.float32:
        raise ValueError("partials must be float32")
    if not (o_parts.is_contiguous() and lse_parts.is_contiguous()):
        raise ValueError("partials must be contiguous")
    if tuple(lse_parts.shape) != tuple(o_parts.shape[:-1]):
        raise ValueError("lse_parts must have the shape of o_parts without its last axis")
    _on_current_device("o_parts", o_parts)
    _same_device(o_parts.device, lse_parts=lse_parts)
    out_dtype = out_dtype or torch.float32
    if o is None:
        o = torch.empty(o_parts.shape[1:], dtype=out_dtype, device=o_parts.device)
    if lse is None:
        lse = torch.empty(lse_parts.shape[1:], dtype=torch.float32, device=o_parts.device)
    if o.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("o must be float32 or bfloat16")
    _need("o", o, o_parts.shape[1:], o.dtype, o_parts.device)
    _need("lse", lse, lse_parts.shape[1:], torch.float32, o_parts.device)
    code = 1 if o.dtype == torch.bfloat16 else 0
    _check(load_library().ra_merge_partials(n, rows, d, _ptr(o_parts), _ptr(lse_parts), _ptr(o), code,
                                            _ptr(lse), _stream(stream)))
    return o, lse


def ra_layout_perm(x, layout, n_shards, inverse=False, seq_dim=None, out=None, stream=None):
    """Natural -> layout order (inverse=False) or back, along ``seq_dim``.

    ``seq_dim`` defaults to 2, the sequence axis of the library's [B, H, S, d] and
    [B, H, S] tensors.  Everything after the sequence axis moves as one row.
    """
    import torch
    if not x.is_contiguous() or not x.is_cuda:
        raise ValueError("x must be a contiguous CUDA tensor")
    seq_dim = (2 if seq_dim is None else seq_dim) % x.dim()
    seq = x.shape[seq_dim]
    outer = int(np.prod(x.shape[:seq_dim], dtype=np.int64)) if seq_dim else 1
    row_bytes = int(np.prod(x.shape[seq_dim + 1:], dtype=np.int64)) * x.element_size()
    if out is None:
        out = torch.empty_like(x)
    _need("out", out, x.shape, x.dtype, x.device)
    _check(load_library().ra_layout_perm(_layout(layout), seq, int(n_shards), int(bool(inverse)), outer,
                                         row_bytes, _ptr(x), _ptr(out), _stream(stream)))
    return out


def ra_layout_index(layout, seq, n_shards):
    """Natural position of every layout-ordered row (host helper)."""
    pos = np.zeros(int(seq), np.int64)
    _check(load_library().ra_layout_index(_layout(layout), int(seq), int(n_shards), pos.ctypes.data))
    return pos


def ra_wait_selftest():
    """Run the tensor-core kernels' bounded wait against a barrier nothing completes
    (about one second); returns the status word it left (2: it gave up as designed)."""
    word = ctypes.c_uint32(0)
    _check(load_library().ra_wait_selftest(ctypes.addressof(word)))
    return word.value


def ra_sync_status(plan, stream=None):
    """Synchronize the stream and raise RaError if a device wait of this plan timed out."""
    _check(load_library().ra_sync_status(plan.handle, _stream(stream)))


def ra_fwd_static(batch, seq, heads_q, heads_kv, n_shards, layout, causal, q, k, v, o=None, lse=None,
                  scale=0.0, stream=None):
    """Fused bf16 forward without a plan and without allocating device memory.

    For callers that must not allocate device memory at run time (the library's
    static scratch array holds the work list).  Returns (O, LSE); pass ``o`` and
    ``lse`` to avoid the two torch allocations this wrapper otherwise makes.
    """
    import torch
    _need("q", q, (batch, heads_q, seq, 128), torch.bfloat16, q.device)
    if not q.is_cuda:
        raise ValueError("q must be a CUDA tensor")
    _need("k", k, (batch, heads_kv, seq, 128), torch.bfloat16, q.device)
    _need("v", v, (batch, heads_kv, seq, 128), torch.bfloat16, q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((batch, heads_q, seq), dtype=torch.float32, device=q.device)
    _need("o", o, q.shape, q.dtype, q.device)
    _need("lse", lse, (batch, heads_q, seq), torch.float32, q.device)
    prob = _Problem(int(batch), int(seq), int(heads_q), int(heads_kv), 128, int(n_shards), _layout(layout),
                    int(bool(causal)), 1, float(scale or 0.0))
    _check(load_library().ra_fwd_static(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                        _stream(stream)))
    return o, lse


def ra_fwd_static_status(stream=None):
    """Raise RaError (RA_ERR_TIMEOUT) if the latest ra_fwd_static call on the current
    device gave up on a device-side wait; synchronizes ``stream`` first."""
    _check(load_library().ra_fwd_static_status(_stream(stream)))


def ra_fwd_step(plan, step, q, k_blk, v_blk, o_part=None, lse_part=None, stream=None):
    """One ring step for every shard over the blocks the shards hold -> (O_t, LSE_t) in float32.

    ``k_blk``/``v_blk`` hold, in the rows of shard p, the block shard p holds at this
    step (K/V themselves at step 0; ``ra_ring_rotate`` passes them on).
    """
    import torch
    pb = plan.problem
    B, Hq, S, d = pb["batch"], pb["heads_q"], pb["seq"], pb["head_dim"]
    _check_qkv(plan, q=q, k_blk=k_blk, v_blk=v_blk)
    _same_device(q.device, k_blk=k_blk, v_blk=v_blk)
    if o_part is None:
        o_part = torch.empty((B, Hq, S, d), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    _need("o_part", o_part, (B, Hq, S, d), torch.float32, q.device)
    _need("lse_part", lse_part, (B, Hq, S), torch.float32, q.device)
    _check(load_library().ra_fwd_step(plan.handle, int(step), _ptr(q), _ptr(k_blk), _ptr(v_blk), _ptr(o_part),
                                      _ptr(lse_part), _stream(stream)))
    return o_part, lse_part


def ra_ring_rotate(plan, k_src, v_src, k_dst=None, v_dst=None, stream=None):
    """Pass every shard's K/V block on to the next shard -> (k_dst, v_dst)."""
    import torch
    _check_qkv(plan, k_src=k_src, v_src=v_src)
    if k_dst is None:
        k_dst = torch.empty_like(k_src)
    if v_dst is None:
        v_dst = torch.empty_like(v_src)
    _check_qkv(plan, k_dst=k_dst, v_dst=v_dst)
    _same_device(k_src.device, v_src=v_src, k_dst=k_dst, v_dst=v_dst)
    _check(load_library().ra_ring_rotate(plan.handle, _ptr(k_src), _ptr(v_src), _ptr(k_dst), _ptr(v_dst),
                                         _stream(stream)))
    return k_dst, v_dst


def ra_ring_fwd(plan, q, k, v, o=None, lse=None, k_buf=None, v_buf=None, o_parts=None, lse_parts=None,
                stream=None, comm_stream=None):
    """Explicit ring driver: N per-step launches, K/V passed on on ``comm_stream``, then a merge.

    Returns (O, LSE).  Scratch (two receive buffers for K and V, the N float32
    partials) is allocated here unless passed in; ``comm_stream`` defaults to a
    new stream (pass the compute stream itself to run without overlap).
    """
    import torch
    pb = plan.problem
    B, Hq, S, d, N = pb["batch"], pb["heads_q"], pb["seq"], pb["head_dim"], pb["n_shards"]
    _check_qkv(plan, q=q, k=k, v=v)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    if N > 1:
        if k_buf is None:
            k_buf = torch.empty((2,) + tuple(k.shape), dtype=k.dtype, device=k.device)
        if v_buf is None:
            v_buf = torch.empty((2,) + tuple(v.shape), dtype=v.dtype, device=v.device)
    if o_parts is None:
        o_parts = torch.empty((N, B, Hq, S, d), dtype=torch.float32, device=q.device)
    if lse_parts is None:
        lse_parts = torch.empty((N, B, Hq, S), dtype=torch.float32, device=q.device)
    _same_device(q.device, k=k, v=v)
    _need("o", o, q.shape, q.dtype, q.device)
    _need("lse", lse, (B, Hq, S), torch.float32, q.device)
    if N > 1:
        _need("k_buf", k_buf, (2,) + tuple(k.shape), k.dtype, q.device)
        _need("v_buf", v_buf, (2,) + tuple(v.shape), v.dtype, q.device)
    _need("o_parts", o_parts, (N, B, Hq, S, d), torch.float32, q.device)
    _need("lse_parts", lse_parts, (N, B, Hq, S), torch.float32, q.device)
    if comm_stream is None:
        comm_stream = torch.cuda.Stream(device=q.device)
    _check(load_library().ra_ring_fwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(k_buf),
                                      _ptr(v_buf), _ptr(o_parts), _ptr(lse_parts), _stream(stream),
                                      _stream(comm_stream)))
    return o, lse


def ra_bwd(plan, q, k, v, o, lse, dout, dq=None, dk=None, dv=None, scratch=None, stream=None):
    """Gradients (dQ, dK, dV) of the forward for the upstream gradient ``dout``.

    ``o`` and ``lse`` are the forward's outputs for the same q, k, v; ``scratch``
    (``ra_bwd_scratch_size`` bytes, float32) is allocated here unless passed in.
    """
    import torch
    pb = plan.problem
    B, Hq, S = pb["batch"], pb["heads_q"], pb["seq"]
    _check_qkv(plan, q=q, k=k, v=v)
    _check_qkv(plan, q=o)
    _check_qkv(plan, q=dout)
    if dq is None:
        dq = torch.empty_like(q)
    if dk is None:
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    if scratch is None:
        scratch = torch.empty(ra_bwd_scratch_size(plan) // 4, dtype=torch.float32, device=q.device)
    elif (scratch.numel() * scratch.element_size() < ra_bwd_scratch_size(plan) or scratch.dtype != torch.float32
          or not scratch.is_contiguous() or scratch.device != q.device):
        raise ValueError("scratch must be a contiguous float32 tensor of at least ra_bwd_scratch_size(plan) "
                         "bytes on the device of q")
    _same_device(q.device, k=k, v=v, o=o, dout=dout)
    _need("lse", lse, (B, Hq, S), torch.float32, q.device)
    _need("dq", dq, q.shape, q.dtype, q.device)
    _need("dk", dk, k.shape, k.dtype, q.device)
    _need("dv", dv, v.shape, v.dtype, q.device)
    _check(load_library().ra_bwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                 _ptr(dq), _ptr(dk), _ptr(dv), _ptr(scratch), _stream(stream)))
    return dq, dk, dv


def ra_bwd_scratch_size(plan):
    """Bytes of the float32 scratch buffer ra_bwd needs for this plan."""
    n = ctypes.c_int64()
    _check(load_library().ra_bwd_scratch_size(plan.handle, ctypes.byref(n)))
    return n.value


def ra_allgather_kv(plan, k, v, k_all=None, v_all=None, stream=None):
    """Gather every shard's K/V block into one natural-order copy -> (k_all, v_all)."""
    import torch
    _check_qkv(plan, k=k, v=v)
    if k_all is None:
        k_all = torch.empty_like(k)
    if v_all is None:
        v_all = torch.empty_like(v)
    _check_qkv(plan, k_all=k_all, v_all=v_all)
    _same_device(k.device, v=v, k_all=k_all, v_all=v_all)
    _check(load_library().ra_allgather_kv(plan.handle, _ptr(k), _ptr(v), _ptr(k_all), _ptr(v_all),
                                          _stream(stream)))
    return k_all, v_all


def ra_fwd_gathered(plan, q, k_all, v_all, o=None, lse=None, stream=None):
    """Forward of the all-gather variant: layout-order q against natural-order K/V -> (O, LSE)."""
    import torch
    pb = plan.problem
    _check_qkv(plan, q=q, k_all=k_all, v_all=v_all)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((pb["batch"], pb["heads_q"], pb["seq"]), dtype=torch.float32, device=q.device)
    _same_device(q.device, k_all=k_all, v_all=v_all)
    _need("o", o, q.shape, q.dtype, q.device)
    _need("lse", lse, (pb["batch"], pb["heads_q"], pb["seq"]), torch.float32, q.device)
    _check(load_library().ra_fwd_gathered(plan.handle, _ptr(q), _ptr(k_all), _ptr(v_all), _ptr(o), _ptr(lse),
                                          _stream(stream)))
    return o, lse


def ra_ulysses_a2a(x, layout, n_shards, direction, out=None, stream=None):
    """Ulysses' exchange.  direction 0: [B, H, S, ...] layout order -> [N, B, H/N, S, ...];
    direction 1: back.  Rows are d = 128 bf16 ([..., 128]) or one float32 ([...])."""
    import torch
    if not x.is_contiguous() or not x.is_cuda:
        raise ValueError("x must be a contiguous CUDA tensor")
    N = int(n_shards)
    if direction == 0:
        B, H, S = x.shape[:3]
        if N < 1 or H % N:
            raise ValueError("the head count must be a multiple of n_shards")
        out_shape = (N, B, H // N, S) + tuple(x.shape[3:])
    else:
        n_, B, hl, S = x.shape[:4]
        if n_ != N:
            raise ValueError(f"x must have n_shards = {N} head shards on its first axis")
        H = hl * N
        out_shape = (B, H, S) + tuple(x.shape[4:])
    row_bytes = int(np.prod(x.shape[3 if direction == 0 else 4:], dtype=np.int64)) * x.element_size()
    if out is None:
        out = torch.empty(out_shape, dtype=x.dtype, device=x.device)
    _need("out", out, out_shape, x.dtype, x.device)
    _check(load_library().ra_ulysses_a2a(int(direction), _layout(layout), int(S), N, int(B), int(H), row_bytes,
                                         _ptr(x), _ptr(out), _stream(stream)))
    return out
