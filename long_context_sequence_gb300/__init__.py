"""Python binding of the Ulysses sequence-parallel attention library (libulysses.so).

Argument marshalling only: every function below forwards to the C entry point of the
same name in include/ulysses.h.  Tensors are torch tensors already on the GPU (their
data pointers are passed); streams default to torch's current stream.  Every step of
the computation runs in the library's CUDA kernels; there is no fallback, and importing
this package fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# ULY_LIBRARY=debug selects the bounds-checking debug build (libulysses_debug.so); any other
# value is taken as the library's path.
_CHOICE = os.environ.get("ULY_LIBRARY", "")
LIB_PATH = (os.path.join(_HERE, "libulysses_debug.so") if _CHOICE == "debug"
            else _CHOICE or os.path.join(_HERE, "libulysses.so"))

(ULY_OK, ULY_ERR_INVALID_ARG, ULY_ERR_UNSUPPORTED, ULY_ERR_CUDA, ULY_ERR_OOM, ULY_ERR_TIMEOUT,
 ULY_ERR_RANGE, ULY_ERR_BOUNDS) = range(8)
ULY_FLAG_INJECT_STALL = 0x1
_STATUS_NAMES = {0: "ULY_OK", 1: "ULY_ERR_INVALID_ARG", 2: "ULY_ERR_UNSUPPORTED",
                 3: "ULY_ERR_CUDA", 4: "ULY_ERR_OOM", 5: "ULY_ERR_TIMEOUT",
                 6: "ULY_ERR_RANGE", 7: "ULY_ERR_BOUNDS"}

EXPORTED = ("ulysses_plan", "ulysses_plan_destroy", "ulysses_workspace_bytes",
            "ulysses_qkv_proj", "ulysses_seq_to_head", "ulysses_seq_to_head_heads",
            "ulysses_attn_fwd", "ulysses_attn_bwd", "ulysses_attn_bwd_noalloc",
            "ulysses_head_to_seq", "ulysses_head_to_seq_qkv", "ulysses_qkv_proj_bwd",
            "ulysses_o_proj", "ulysses_o_proj_bwd", "ulysses_ring_workspace_bytes",
            "ulysses_ring_attn_fwd", "ulysses_ring_volume",
            "ulysses_sync_status", "ulysses_bytes_moved", "ulysses_a2a_volume",
            "ulysses_last_error", "ulysses_plan_rank", "ulysses_a2a_table",
            "ulysses_a2a_pack_qkv", "ulysses_a2a_pack_heads", "ulysses_a2a_unpack_heads",
            "ulysses_a2a_unpack_qkv", "ulysses_a2a_exchange", "ulysses_nccl_unique_id",
            "ulysses_nccl_comm_init", "ulysses_nccl_comm_destroy")


class UlyssesError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (_STATUS_NAMES.get(status, str(status)), message))
        self.status = status


class UlyConfig(ctypes.Structure):
    """Mirror of struct uly_config."""
    _fields_ = [("seq_len", ctypes.c_int64), ("batch", ctypes.c_int32), ("P", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("causal", ctypes.c_int32), ("wait_timeout_ms", ctypes.c_int32),
                ("softmax_scale", ctypes.c_double), ("rope_theta", ctypes.c_double),
                ("flags", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


class A2ABlock(ctypes.Structure):
    """Mirror of struct uly_a2a_block."""
    _fields_ = [("peer", ctypes.c_int32), ("n_tokens", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("send_token_begin", ctypes.c_int64), ("recv_token_begin", ctypes.c_int64),
                ("send_head_begin", ctypes.c_int32), ("recv_head_begin", ctypes.c_int32),
                ("send_offset", ctypes.c_uint64), ("recv_offset", ctypes.c_uint64),
                ("count", ctypes.c_uint64)]


def make_config(seq_len, P, hidden, n_q_heads, n_kv_heads, head_dim, rope_theta=0.0,
                softmax_scale=0.0, flags=0, wait_timeout_ms=0) -> UlyConfig:
    return UlyConfig(seq_len=seq_len, batch=1, P=P, hidden=hidden, n_q_heads=n_q_heads,
                     n_kv_heads=n_kv_heads, head_dim=head_dim, causal=1,
                     wait_timeout_ms=wait_timeout_ms, softmax_scale=softmax_scale,
                     rope_theta=rope_theta, flags=flags, reserved=0)


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libulysses.so and declare its signatures (no GPU needed)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError("libulysses.so is not built (%s); run __graft_entry__.build() or "
                          "python long_context_sequence_gb300/build.py" % path)
    lib = ctypes.CDLL(path)
    vp, i32, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64
    sig = {
        "ulysses_plan": ([ctypes.POINTER(UlyConfig), ctypes.POINTER(vp)], i32),
        "ulysses_plan_destroy": ([vp], i32),
        "ulysses_workspace_bytes": ([vp], ctypes.c_size_t),
        "ulysses_qkv_proj": ([vp, vp, vp, vp, vp], i32),
        "ulysses_seq_to_head": ([vp, vp, i32, i32, vp, vp, vp, vp], i32),
        "ulysses_seq_to_head_heads": ([vp, vp, i32, vp, vp], i32),
        "ulysses_attn_fwd": ([vp] * 8, i32),
        "ulysses_attn_bwd": ([vp] * 13, i32),
        "ulysses_attn_bwd_noalloc": ([vp] * 12, i32),
        "ulysses_head_to_seq": ([vp, vp, i32, vp, vp], i32),
        "ulysses_head_to_seq_qkv": ([vp, vp, vp, vp, i32, vp, vp], i32),
        "ulysses_qkv_proj_bwd": ([vp] * 7, i32),
        "ulysses_o_proj": ([vp] * 5, i32),
        "ulysses_o_proj_bwd": ([vp] * 7, i32),
        "ulysses_ring_workspace_bytes": ([vp], ctypes.c_size_t),
        "ulysses_ring_attn_fwd": ([vp] * 8, i32),
        "ulysses_ring_volume": ([ctypes.POINTER(UlyConfig), ctypes.POINTER(u64)], i32),
        "ulysses_sync_status": ([vp, vp], i32),
        "ulysses_bytes_moved": ([vp], u64),
        "ulysses_a2a_volume": ([ctypes.POINTER(UlyConfig), ctypes.POINTER(u64),
                                ctypes.POINTER(u64)], i32),
        "ulysses_last_error": ([], ctypes.c_char_p),
        "ulysses_plan_rank": ([ctypes.POINTER(UlyConfig), ctypes.c_int32, ctypes.POINTER(vp)], i32),
        "ulysses_a2a_table": ([ctypes.POINTER(UlyConfig), ctypes.c_int32, ctypes.c_int32,
                               ctypes.c_int32, ctypes.POINTER(A2ABlock)], i32),
        "ulysses_a2a_pack_qkv": ([vp, vp, i32, i32, vp, vp, vp, vp], i32),
        "ulysses_a2a_pack_heads": ([vp, vp, i32, vp, vp], i32),
        "ulysses_a2a_unpack_heads": ([vp, vp, i32, vp, vp], i32),
        "ulysses_a2a_unpack_qkv": ([vp, vp, vp, vp, i32, vp, vp], i32),
        "ulysses_a2a_exchange": ([vp, vp, ctypes.c_int32, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                  ctypes.POINTER(u64), vp], i32),
        "ulysses_nccl_unique_id": ([ctypes.POINTER(ctypes.c_uint8)], i32),
        "ulysses_nccl_comm_init": ([ctypes.c_int32, ctypes.c_int32,
                                    ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(vp)], i32),
        "ulysses_nccl_comm_destroy": ([vp], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(status: int):
    if status != ULY_OK:
        raise UlyssesError(status, load_library().ulysses_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("tensor must be on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """Owns a uly_plan handle (rank is None for the single-GPU virtual ranks)."""

    def __init__(self, handle: int, cfg: UlyConfig, rank=None):
        self.handle = handle
        self.cfg = cfg
        self.rank = rank

    def close(self):
        if self.handle:
            _check(load_library().ulysses_plan_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # shapes of the tensors of one block (see include/ulysses.h)
    def shapes(self):
        c = self.cfg
        S, P, H, G, D = c.seq_len, c.P, c.n_q_heads, c.n_kv_heads, c.head_dim
        if self.rank is not None:       # one real rank: its shard and its head group
            n, hl, gl = S // P, H // P, G // P
            return {"x": (n, c.hidden), "w": ((H + 2 * G) * D, c.hidden),
                    "qkv": (n, H + 2 * G, D), "q": (P, n, hl, D), "k": (P, n, gl, D),
                    "v": (P, n, gl, D), "o": (P, n, hl, D), "lse": (hl, S),
                    "o_seq": (n, H, D)}
        return {"x": (S, c.hidden), "w": ((H + 2 * G) * D, c.hidden),
                "qkv": (P, S // P, H + 2 * G, D), "q": (P, S, H // P, D),
                "k": (P, S, G // P, D), "v": (P, S, G // P, D), "o": (P, S, H // P, D),
                "lse": (P, H // P, S), "o_seq": (P, S // P, H, D),
                "kv_seq": (P, S // P, G, D)}


def ulysses_plan(cfg: UlyConfig) -> Plan:
    h = ctypes.c_void_p()
    _check(load_library().ulysses_plan(ctypes.byref(cfg), ctypes.byref(h)))
    return Plan(h.value, cfg)


def ulysses_plan_rank(cfg: UlyConfig, rank: int) -> Plan:
    """Plan of one real rank of a cfg.P-GPU group."""
    h = ctypes.c_void_p()
    _check(load_library().ulysses_plan_rank(ctypes.byref(cfg), int(rank), ctypes.byref(h)))
    return Plan(h.value, cfg, rank=int(rank))


def ulysses_a2a_table(cfg: UlyConfig, rank: int, to_head: bool, n_heads: int):
    """The all-to-all block table of `rank` (host only): one dict per peer."""
    blocks = (A2ABlock * cfg.P)()
    _check(load_library().ulysses_a2a_table(ctypes.byref(cfg), int(rank), 1 if to_head else 0,
                                            int(n_heads), blocks))
    return [{f: getattr(b, f) for f, _ in A2ABlock._fields_ if f != "reserved"} for b in blocks]


def ulysses_a2a_pack_qkv(plan, qkv_local, send_q, send_k, send_v, apply_rope=False,
                         stream=None):
    import torch
    in_fp32 = 1 if qkv_local.dtype == torch.float32 else 0
    _check(load_library().ulysses_a2a_pack_qkv(plan.handle, _ptr(qkv_local), in_fp32,
                                               1 if apply_rope else 0, _ptr(send_q),
                                               _ptr(send_k), _ptr(send_v), _stream(stream)))


def ulysses_a2a_pack_heads(plan, x_local, n_heads, send, stream=None):
    _check(load_library().ulysses_a2a_pack_heads(plan.handle, _ptr(x_local), int(n_heads),
                                                 _ptr(send), _stream(stream)))


def ulysses_a2a_unpack_heads(plan, recv, n_heads, x_local, stream=None):
    _check(load_library().ulysses_a2a_unpack_heads(plan.handle, _ptr(recv), int(n_heads),
                                                   _ptr(x_local), _stream(stream)))


def ulysses_a2a_unpack_qkv(plan, recv_dq, recv_dk, recv_dv, dqkv_local, apply_rope=False,
                           stream=None):
    _check(load_library().ulysses_a2a_unpack_qkv(plan.handle, _ptr(recv_dq), _ptr(recv_dk),
                                                 _ptr(recv_dv), 1 if apply_rope else 0,
                                                 _ptr(dqkv_local), _stream(stream)))


def ulysses_a2a_exchange(plan, comm, sends, recvs, stream=None):
    """The all-to-all of block-major buffers (one NCCL group over all pairs)."""
    n = len(sends)
    if n != len(recvs) or n == 0:
        raise ValueError("need as many receive buffers as send buffers")
    for a, b in zip(sends, recvs):
        if a.nbytes != b.nbytes or a.nbytes % plan.cfg.P:
            raise ValueError("send and receive buffers must have equal sizes divisible by P")
    sp = (ctypes.c_void_p * n)(*[_ptr(t) for t in sends])
    rp = (ctypes.c_void_p * n)(*[_ptr(t) for t in recvs])
    bp = (ctypes.c_uint64 * n)(*[t.nbytes // plan.cfg.P for t in sends])
    _check(load_library().ulysses_a2a_exchange(plan.handle, comm, n, sp, rp, bp,
                                               _stream(stream)))


def ulysses_nccl_unique_id() -> bytes:
    buf = (ctypes.c_uint8 * 128)()
    _check(load_library().ulysses_nccl_unique_id(buf))
    return bytes(buf)


def ulysses_nccl_comm_init(nranks: int, rank: int, uid: bytes) -> int:
    """Joins an NCCL communicator (all nranks processes call it, each on its own GPU)."""
    if len(uid) != 128:
        raise ValueError("the NCCL id has 128 bytes")
    buf = (ctypes.c_uint8 * 128)(*uid)
    comm = ctypes.c_void_p()
    _check(load_library().ulysses_nccl_comm_init(int(nranks), int(rank), buf, ctypes.byref(comm)))
    return comm.value


def ulysses_nccl_comm_destroy(comm: int):
    _check(load_library().ulysses_nccl_comm_destroy(comm))


def ulysses_plan_destroy(plan: Plan):
    plan.close()


def ulysses_workspace_bytes(plan: Plan) -> int:
    return int(load_library().ulysses_workspace_bytes(plan.handle))


def ulysses_qkv_proj(plan, x, w, qkv, stream=None):
    _check(load_library().ulysses_qkv_proj(plan.handle, _ptr(x), _ptr(w), _ptr(qkv),
                                           _stream(stream)))


def ulysses_seq_to_head(plan, qkv_seq, q, k, v, apply_rope=False, stream=None):
    import torch
    in_fp32 = 1 if qkv_seq.dtype == torch.float32 else 0
    _check(load_library().ulysses_seq_to_head(plan.handle, _ptr(qkv_seq), in_fp32,
                                              1 if apply_rope else 0, _ptr(q), _ptr(k), _ptr(v),
                                              _stream(stream)))


def ulysses_seq_to_head_heads(plan, x_seq, n_heads, x_head, stream=None):
    _check(load_library().ulysses_seq_to_head_heads(plan.handle, _ptr(x_seq), int(n_heads),
                                                    _ptr(x_head), _stream(stream)))


def ulysses_attn_fwd(plan, q, k, v, o, lse, stream=None, o_lo=None):
    _check(load_library().ulysses_attn_fwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                           _ptr(o_lo), _ptr(lse), _stream(stream)))


def ulysses_attn_bwd(plan, q, k, v, o, lse, d_o, dq, dk, dv, workspace, stream=None,
                     o_lo=None):
    _check(load_library().ulysses_attn_bwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                           _ptr(o_lo), _ptr(lse), _ptr(d_o), _ptr(dq),
                                           _ptr(dk), _ptr(dv), _ptr(workspace),
                                           _stream(stream)))


def ulysses_attn_bwd_noalloc(plan, q, k, v, o, lse, d_o, dq, dk, dv, stream=None, o_lo=None):
    """The backward with the library's fixed device scratch instead of a workspace."""
    _check(load_library().ulysses_attn_bwd_noalloc(plan.handle, _ptr(q), _ptr(k), _ptr(v),
                                                   _ptr(o), _ptr(o_lo), _ptr(lse), _ptr(d_o),
                                                   _ptr(dq), _ptr(dk), _ptr(dv),
                                                   _stream(stream)))


def ulysses_head_to_seq(plan, x_head, n_heads, x_seq, stream=None):
    _check(load_library().ulysses_head_to_seq(plan.handle, _ptr(x_head), int(n_heads),
                                              _ptr(x_seq), _stream(stream)))


def ulysses_head_to_seq_qkv(plan, dq, dk, dv, dqkv_seq, apply_rope=False, stream=None):
    _check(load_library().ulysses_head_to_seq_qkv(plan.handle, _ptr(dq), _ptr(dk), _ptr(dv),
                                                  1 if apply_rope else 0, _ptr(dqkv_seq),
                                                  _stream(stream)))


def ulysses_qkv_proj_bwd(plan, x, w, dqkv, dx=None, dw=None, stream=None):
    _check(load_library().ulysses_qkv_proj_bwd(plan.handle, _ptr(x), _ptr(w), _ptr(dqkv),
                                               _ptr(dx), _ptr(dw), _stream(stream)))


def ulysses_o_proj(plan, o_head, wo, y, stream=None):
    _check(load_library().ulysses_o_proj(plan.handle, _ptr(o_head), _ptr(wo), _ptr(y),
                                         _stream(stream)))


def ulysses_o_proj_bwd(plan, o_head, wo, dy, do_head=None, dwo=None, stream=None):
    _check(load_library().ulysses_o_proj_bwd(plan.handle, _ptr(o_head), _ptr(wo), _ptr(dy),
                                             _ptr(do_head), _ptr(dwo), _stream(stream)))


def ulysses_sync_status(plan, stream=None) -> int:
    """Returns the device status (ULY_OK or an error code) instead of raising."""
    return int(load_library().ulysses_sync_status(plan.handle, _stream(stream)))


def ulysses_bytes_moved(plan) -> int:
    return int(load_library().ulysses_bytes_moved(plan.handle))


def ulysses_a2a_volume(cfg: UlyConfig):
    a, b = ctypes.c_uint64(), ctypes.c_uint64()
    _check(load_library().ulysses_a2a_volume(ctypes.byref(cfg), ctypes.byref(a), ctypes.byref(b)))
    return int(a.value), int(b.value)


def ulysses_ring_workspace_bytes(plan) -> int:
    return int(load_library().ulysses_ring_workspace_bytes(plan.handle))


def ulysses_ring_attn_fwd(plan, q_seq, k_seq, v_seq, o_seq, lse, workspace, stream=None):
    _check(load_library().ulysses_ring_attn_fwd(plan.handle, _ptr(q_seq), _ptr(k_seq),
                                                _ptr(v_seq), _ptr(o_seq), _ptr(lse),
                                                _ptr(workspace), _stream(stream)))


def ulysses_ring_volume(cfg: UlyConfig) -> int:
    a = ctypes.c_uint64()
    _check(load_library().ulysses_ring_volume(ctypes.byref(cfg), ctypes.byref(a)))
    return int(a.value)


def ulysses_last_error() -> str:
    return load_library().ulysses_last_error().decode()
