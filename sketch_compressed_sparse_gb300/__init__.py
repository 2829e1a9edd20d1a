"""Python binding of libs2, the sm_103a S2 Reducer hot path.

Argument marshalling only: every function below checks the torch tensors it
is given (device, dtype, contiguity, sizes), passes their device pointers and
the current CUDA stream to the C ABI declared in ``include/s2.h``, and raises
``S2Error`` on a non-OK status. All computation happens in the CUDA kernels
of ``libs2.so``; there is no fallback. The library is loaded by the first
call; if it has not been built that call raises ``ImportError`` (build it
with ``python -m sketch_compressed_sparse_gb300.build``).

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

__all__ = [
    "S2Error",
    "lib_path",
    "nwords",
    "s2_encode",
    "s2_encode_batched",
    "s2_encode_batched_path",
    "S2_PATH_AUTO",
    "S2_PATH_L2",
    "S2_PATH_SMEM",
    "S2_SMEM_SKETCH_MAX_BYTES",
    "s2_reduce",
    "s2_encode_reduce_fused",
    "s2_encode_batched_blocks",
    "s2_block_topk",
    "s2_sparse_pack",
    "s2_sparse_sum",
    "s2_block_topk_workspace_size",
    "s2_decode_dense_blocks",
    "s2_decode_dense",
    "s2_decode_workspace_size",
    "s2_decode_dense_workspace_size",
    "s2_decode_dense_ws",
    "s2_decode_compact",
    "s2_decode_compact_noalloc",
    "s2_hash",
    "s2_pipeline_workspace_size",
    "s2_pipeline_dense_host",
    "s2_status_string",
    "s2_version",
    "S2_F32",
    "S2_BF16",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libs2.so")

S2_OK, S2_ERR_INVALID_ARG, S2_ERR_ALIGNMENT, S2_ERR_UNSUPPORTED, S2_ERR_CUDA = range(5)
S2_F32, S2_BF16 = 0, 1


class Params(ctypes.Structure):
    _fields_ = [("d", ctypes.c_uint32), ("w", ctypes.c_uint32), ("seed", ctypes.c_uint32)]


_u32, _u64, _i32, _f32, _vp, _sz = (ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int, ctypes.c_float,
                                     ctypes.c_void_p, ctypes.c_size_t)

_SIGS = {
    "s2_encode": ([_vp, _i32, _u64, Params, _vp, _vp, _vp], _i32),
    "s2_encode_batched": ([_vp, _i32, _u32, _u64, Params, _vp, _vp, _vp], _i32),
    "s2_encode_batched_path": ([_vp, _i32, _u32, _u64, Params, _i32, _vp, _vp, _vp], _i32),

    "s2_reduce": ([_vp, _vp, _u32, _u64, Params, _vp, _vp, _vp], _i32),
    "s2_encode_reduce_fused": ([_vp, _i32, _u32, _u64, Params, _vp, _vp, _vp], _i32),
    "s2_encode_batched_blocks": ([_vp, _i32, _u32, _u64, _u32, Params, _vp, _vp, _vp], _i32),
    "s2_block_topk_workspace_size": ([_u32, _u64, _u32, ctypes.POINTER(_sz)], _i32),
    "s2_sparse_pack_workspace_size": ([_u32, _u64, ctypes.POINTER(_sz)], _i32),
    "s2_sparse_pack": ([_vp, _u32, _u64, _vp, _vp, _u64, _vp, _vp, _sz, _vp], _i32),
    "s2_sparse_sum": ([_vp, _vp, _vp, _u32, _u64, _u64, _vp, _vp], _i32),
    "s2_block_topk": ([_vp, _vp, _u32, _u64, _u32, _u64, _vp, _vp, _sz, _vp], _i32),
    "s2_decode_dense_blocks": ([_vp, _vp, _u64, _u32, Params, _f32, _vp, _vp], _i32),
    "s2_decode_dense": ([_vp, _vp, _u64, Params, _f32, _vp, _vp], _i32),
    "s2_decode_workspace_size": ([_u64, ctypes.POINTER(_sz)], _i32),
    "s2_decode_dense_workspace_size": ([_u64, Params, ctypes.POINTER(_sz)], _i32),
    "s2_decode_dense_ws": ([_vp, _vp, _u64, Params, _f32, _vp, _vp, _sz, _vp], _i32),
    "s2_decode_compact": ([_vp, _vp, _u64, Params, _f32, _vp, _vp, _u64, _vp, _vp, _sz, _vp], _i32),
    "s2_decode_compact_noalloc": ([_vp, _vp, _u64, Params, _f32, _vp, _vp, _u64, _vp, _vp], _i32),
    "s2_hash": ([_vp, _u64, Params, _vp, _vp, _vp], _i32),
    "s2_pipeline_workspace_size": ([_i32, _u32, _u64, Params, ctypes.POINTER(_sz)], _i32),
    "s2_pipeline_dense_host": ([_vp, _i32, _u32, _u64, Params, _f32, _vp, _vp, _sz, _vp], _i32),
    "s2_status_string": ([_i32], ctypes.c_char_p),
    "s2_version": ([], ctypes.c_char_p),
}
_fns = {}


def _load():
    """Load libs2.so once; raise ImportError if it has not been built."""
    if _fns:
        return _fns
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"libs2.so not found at {_LIB_PATH}: build the CUDA library first "
            "(python -m sketch_compressed_sparse_gb300.build)")
    lib = ctypes.CDLL(_LIB_PATH)
    for name, (args, res) in _SIGS.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
        _fns[name] = f
    return _fns


def _f(name):
    return (_fns or _load())[name]


class S2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {s2_status_string(status)} ({status})")


def lib_path() -> str:
    """Path of the loaded libs2.so (loads it; ImportError if not built)."""
    _load()
    return _LIB_PATH


def s2_status_string(status: int) -> str:
    return _f("s2_status_string")(status).decode()


def s2_version() -> str:
    return _f("s2_version")().decode()


def nwords(n: int) -> int:
    return (n + 31) // 32


def _check(status: int, where: str):
    if status != S2_OK:
        raise S2Error(status, where)


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dev(t: Optional[torch.Tensor], name: str, dtypes, numel: Optional[int] = None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {numel}")
    return t.data_ptr() if t.numel() else None


_U32 = (torch.int32, torch.uint32) if hasattr(torch, "uint32") else (torch.int32,)
_GRAD = (torch.float32, torch.bfloat16)


def _dtype_code(g: torch.Tensor) -> int:
    return S2_F32 if g.dtype == torch.float32 else S2_BF16


def s2_encode(grad: torch.Tensor, d: int, w: int, seed: int, bitmap: torch.Tensor, sketch: torch.Tensor,
              stream=None) -> None:
    """One worker: grad [n] -> bitmap [nw] (int32 words), sketch [d, w] float32."""
    n = grad.numel()
    _check(_f("s2_encode")(_dev(grad, "grad", _GRAD), _dtype_code(grad), n, Params(d, w, seed),
                _dev(bitmap, "bitmap", _U32, nwords(n)), _dev(sketch, "sketch", (torch.float32,), d * w),
                _stream(stream)), "s2_encode")


def s2_encode_batched(grad: torch.Tensor, d: int, w: int, seed: int, bitmaps: torch.Tensor,
                      sketches: torch.Tensor, stream=None) -> None:
    """W workers: grad [W, n] -> bitmaps [W, nw], sketches [W, d, w]."""
    if grad.dim() != 2:
        raise ValueError("grad must be [W, n]")
    W, n = grad.shape
    _check(_f("s2_encode_batched")(_dev(grad, "grad", _GRAD), _dtype_code(grad), W, n, Params(d, w, seed),
                 _dev(bitmaps, "bitmaps", _U32, W * nwords(n)),
                 _dev(sketches, "sketches", (torch.float32,), W * d * w), _stream(stream)), "s2_encode_batched")


S2_PATH_AUTO, S2_PATH_L2, S2_PATH_SMEM = 0, 1, 2
S2_SMEM_SKETCH_MAX_BYTES = 192 * 1024
_PATHS = {"auto": S2_PATH_AUTO, "l2": S2_PATH_L2, "smem": S2_PATH_SMEM}


def s2_encode_batched_path(grad: torch.Tensor, d: int, w: int, seed: int, bitmaps: torch.Tensor,
                           sketches: torch.Tensor, path="auto", stream=None) -> None:
    """s2_encode_batched with the accumulation path: "auto", "l2" or "smem"
    (a per-block copy of the sketch in shared memory; 4*d*w must be at most
    S2_SMEM_SKETCH_MAX_BYTES)."""
    if grad.dim() != 2:
        raise ValueError("grad must be [W, n]")
    code = _PATHS[path] if isinstance(path, str) else int(path)
    W, n = grad.shape
    _check(_f("s2_encode_batched_path")(_dev(grad, "grad", _GRAD), _dtype_code(grad), W, n, Params(d, w, seed),
                                        code, _dev(bitmaps, "bitmaps", _U32, W * nwords(n)),
                                        _dev(sketches, "sketches", (torch.float32,), W * d * w), _stream(stream)),
           "s2_encode_batched_path")


def s2_reduce(bitmaps: torch.Tensor, sketches: torch.Tensor, n: int, d: int, w: int, bitmap_out: torch.Tensor,
              sketch_out: torch.Tensor, stream=None) -> None:
    """bitmaps [W, nw], sketches [W, d, w] -> bitmap_out [nw] (OR), sketch_out [d, w] (sum)."""
    W = sketches.shape[0] if sketches.dim() == 3 else sketches.numel() // max(d * w, 1)
    _check(_f("s2_reduce")(_dev(bitmaps, "bitmaps", _U32, W * nwords(n)),
                _dev(sketches, "sketches", (torch.float32,), W * d * w), W, n, Params(d, w, 0),
                _dev(bitmap_out, "bitmap_out", _U32, nwords(n)),
                _dev(sketch_out, "sketch_out", (torch.float32,), d * w), _stream(stream)), "s2_reduce")


def s2_encode_reduce_fused(grad: torch.Tensor, d: int, w: int, seed: int, bitmap_out: torch.Tensor,
                           sketch_out: torch.Tensor, stream=None) -> None:
    """W resident workers in one pass: grad [W, n] -> aggregate bitmap [nw], summed sketch [d, w]."""
    if grad.dim() != 2:
        raise ValueError("grad must be [W, n]")
    W, n = grad.shape
    _check(_f("s2_encode_reduce_fused")(_dev(grad, "grad", _GRAD), _dtype_code(grad), W, n, Params(d, w, seed),
                                        _dev(bitmap_out, "bitmap_out", _U32, nwords(n)),
                                        _dev(sketch_out, "sketch_out", (torch.float32,), d * w), _stream(stream)),
           "s2_encode_reduce_fused")


def s2_block_topk_workspace_size(W: int, n: int, block: int) -> int:
    b = _sz()
    _check(_f("s2_block_topk_workspace_size")(W, n, block, ctypes.byref(b)), "s2_block_topk_workspace_size")
    return int(b.value)


def s2_block_topk(grad: torch.Tensor, residual: torch.Tensor, block: int, K: int, sparse_out: torch.Tensor,
                  workspace: torch.Tensor, stream=None) -> None:
    """Block-wise Top-K with error feedback: grad [W, n], residual [W, n] (in/out) -> sparse_out [W, n]."""
    if grad.dim() != 2:
        raise ValueError("grad must be [W, n]")
    W, n = grad.shape
    _check(_f("s2_block_topk")(_dev(grad, "grad", (torch.float32,), W * n),
                               _dev(residual, "residual", (torch.float32,), W * n), W, n, block, K,
                               _dev(sparse_out, "sparse_out", (torch.float32,), W * n),
                               _dev(workspace, "workspace", (torch.uint8,)), workspace.numel(), _stream(stream)),
           "s2_block_topk")


def s2_sparse_pack_workspace_size(W: int, n: int) -> int:
    b = _sz()
    _check(_f("s2_sparse_pack_workspace_size")(W, n, ctypes.byref(b)), "s2_sparse_pack_workspace_size")
    return int(b.value)


def s2_sparse_pack(grad: torch.Tensor, idx_out: torch.Tensor, val_out: torch.Tensor, counts_out: torch.Tensor,
                   workspace: torch.Tensor, stream=None) -> None:
    """AllGather baseline, pack: grad [W, n] -> idx_out/val_out [W, cap] (ascending), counts_out [W] int64."""
    W, n = grad.shape
    cap = idx_out.shape[1] if idx_out.dim() == 2 else 0
    _check(_f("s2_sparse_pack")(_dev(grad, "grad", (torch.float32,), W * n), W, n,
                                _dev(idx_out, "idx_out", _U32, W * cap), _dev(val_out, "val_out", (torch.float32,), W * cap),
                                cap, _dev(counts_out, "counts_out", (torch.int64,), W),
                                _dev(workspace, "workspace", (torch.uint8,)), workspace.numel(), _stream(stream)),
           "s2_sparse_pack")


def s2_sparse_sum(idx: torch.Tensor, val: torch.Tensor, counts: torch.Tensor, n: int, out: torch.Tensor,
                  stream=None) -> None:
    """AllGather baseline, sum: the W gathered lists -> out [n] (worker order 0..W-1)."""
    W, cap = idx.shape
    _check(_f("s2_sparse_sum")(_dev(idx, "idx", _U32, W * cap), _dev(val, "val", (torch.float32,), W * cap),
                               _dev(counts, "counts", (torch.int64,), W), W, cap, n,
                               _dev(out, "out", (torch.float32,), n), _stream(stream)), "s2_sparse_sum")


def nblockwords(n: int, block: int) -> int:
    return nwords((n + block - 1) // block)


def s2_encode_batched_blocks(grad: torch.Tensor, block: int, d: int, w: int, seed: int, block_bitmaps: torch.Tensor,
                             sketches: torch.Tensor, stream=None) -> None:
    """W workers, one bitmap bit per block: grad [W, n] -> block_bitmaps [W, nbw], sketches [W, d, w]."""
    if grad.dim() != 2:
        raise ValueError("grad must be [W, n]")
    W, n = grad.shape
    _check(_f("s2_encode_batched_blocks")(_dev(grad, "grad", _GRAD), _dtype_code(grad), W, n, block,
                                          Params(d, w, seed),
                                          _dev(block_bitmaps, "block_bitmaps", _U32, W * nblockwords(n, block)),
                                          _dev(sketches, "sketches", (torch.float32,), W * d * w), _stream(stream)),
           "s2_encode_batched_blocks")


def s2_decode_dense_blocks(block_bitmap: torch.Tensor, sketch: torch.Tensor, n: int, block: int, d: int, w: int,
                           seed: int, out: torch.Tensor, scale: float = 1.0, stream=None) -> None:
    """Decode every position of every marked block: block_bitmap [nbw], sketch [d, w] -> out [n]."""
    _check(_f("s2_decode_dense_blocks")(_dev(block_bitmap, "block_bitmap", _U32, nblockwords(n, block)),
                                        _dev(sketch, "sketch", (torch.float32,), d * w), n, block,
                                        Params(d, w, seed), scale, _dev(out, "out", (torch.float32,), n),
                                        _stream(stream)), "s2_decode_dense_blocks")


def s2_decode_dense(bitmap: torch.Tensor, sketch: torch.Tensor, n: int, d: int, w: int, seed: int,
                    out: torch.Tensor, scale: float = 1.0, stream=None) -> None:
    """bitmap [nw], sketch [d, w] -> out [n] float32 (median estimates, +0.0 at unset bits)."""
    _check(_f("s2_decode_dense")(_dev(bitmap, "bitmap", _U32, nwords(n)), _dev(sketch, "sketch", (torch.float32,), d * w), n,
                 Params(d, w, seed), scale, _dev(out, "out", (torch.float32,), n), _stream(stream)),
           "s2_decode_dense")


def s2_decode_dense_workspace_size(n: int, d: int, w: int) -> int:
    b = _sz()
    _check(_f("s2_decode_dense_workspace_size")(n, Params(d, w, 0), ctypes.byref(b)), "s2_decode_dense_workspace_size")
    return int(b.value)


def s2_decode_dense_ws(bitmap: torch.Tensor, sketch: torch.Tensor, n: int, d: int, w: int, seed: int,
                       out: torch.Tensor, workspace: torch.Tensor, scale: float = 1.0, stream=None) -> None:
    """s2_decode_dense with a workspace (the row-pass median for sketches larger than L2 can hold)."""
    _check(_f("s2_decode_dense_ws")(_dev(bitmap, "bitmap", _U32, nwords(n)), _dev(sketch, "sketch", (torch.float32,), d * w),
                                    n, Params(d, w, seed), scale, _dev(out, "out", (torch.float32,), n),
                                    _dev(workspace, "workspace", (torch.uint8,)), workspace.numel(), _stream(stream)),
           "s2_decode_dense_ws")


def s2_decode_workspace_size(n: int) -> int:
    b = _sz()
    _check(_f("s2_decode_workspace_size")(n, ctypes.byref(b)), "s2_decode_workspace_size")
    return int(b.value)


def s2_decode_compact(bitmap: torch.Tensor, sketch: torch.Tensor, n: int, d: int, w: int, seed: int,
                      idx_out: torch.Tensor, val_out: torch.Tensor, count_out: torch.Tensor,
                      workspace: torch.Tensor, scale: float = 1.0, stream=None) -> None:
    """bitmap, sketch -> idx_out [cap] int32, val_out [cap] float32, count_out [1] int64 (device)."""
    cap = min(idx_out.numel(), val_out.numel())
    _check(_f("s2_decode_compact")(_dev(bitmap, "bitmap", _U32, nwords(n)), _dev(sketch, "sketch", (torch.float32,), d * w), n,
                 Params(d, w, seed), scale, _dev(idx_out, "idx_out", _U32), _dev(val_out, "val_out", (torch.float32,)),
                 cap, _dev(count_out, "count_out", (torch.int64,), 1), _dev(workspace, "workspace", (torch.uint8,)),
                 workspace.numel(), _stream(stream)), "s2_decode_compact")


def s2_decode_compact_noalloc(bitmap: torch.Tensor, sketch: torch.Tensor, n: int, d: int, w: int, seed: int,
                              idx_out: torch.Tensor, val_out: torch.Tensor, count_out: torch.Tensor,
                              scale: float = 1.0, stream=None) -> None:
    """s2_decode_compact with the library's own scratch instead of a workspace (n <= 2^30).

    For callers that cannot allocate a workspace; see include/s2.h for the
    one-time set-up on a device and why overlapping calls must be avoided.
    """
    cap = min(idx_out.numel(), val_out.numel())
    _check(_f("s2_decode_compact_noalloc")(
        _dev(bitmap, "bitmap", _U32, nwords(n)), _dev(sketch, "sketch", (torch.float32,), d * w), n,
        Params(d, w, seed), scale, _dev(idx_out, "idx_out", _U32), _dev(val_out, "val_out", (torch.float32,)),
        cap, _dev(count_out, "count_out", (torch.int64,), 1), _stream(stream)), "s2_decode_compact_noalloc")


def s2_hash(idx: torch.Tensor, d: int, w: int, seed: int, bucket_out: torch.Tensor, sign_out: torch.Tensor,
            stream=None) -> None:
    """idx [m] -> bucket_out [d, m] int32, sign_out [d, m] int8."""
    m = idx.numel()
    _check(_f("s2_hash")(_dev(idx, "idx", _U32), m, Params(d, w, seed), _dev(bucket_out, "bucket_out", _U32, d * m),
                 _dev(sign_out, "sign_out", (torch.int8,), d * m), _stream(stream)), "s2_hash")


def s2_pipeline_workspace_size(dtype: torch.dtype, W: int, n: int, d: int, w: int) -> int:
    b = _sz()
    _check(_f("s2_pipeline_workspace_size")(S2_F32 if dtype == torch.float32 else S2_BF16, W, n, Params(d, w, 0), ctypes.byref(b)),
           "s2_pipeline_workspace_size")
    return int(b.value)


def s2_pipeline_dense_host(host_grad: torch.Tensor, d: int, w: int, seed: int, host_out: torch.Tensor,
                           workspace: torch.Tensor, scale: float = 1.0, stream=None) -> None:
    """HOST grad [W, n] -> HOST out [n]; queued on the stream. Pinned tensors
    are read / written in place by the kernels; pageable ones are staged."""
    if host_grad.is_cuda or host_out.is_cuda:
        raise ValueError("s2_pipeline_dense_host takes host tensors")
    if host_grad.dim() != 2 or host_grad.dtype not in _GRAD or not host_grad.is_contiguous():
        raise ValueError("host_grad must be a contiguous [W, n] float32/bfloat16 tensor")
    W, n = host_grad.shape
    if host_out.dtype != torch.float32 or host_out.numel() < n or not host_out.is_contiguous():
        raise ValueError("host_out must be a contiguous float32 tensor of n elements")
    _check(_f("s2_pipeline_dense_host")(host_grad.data_ptr(), _dtype_code(host_grad), W, n, Params(d, w, seed), scale,
                 host_out.data_ptr(), _dev(workspace, "workspace", (torch.uint8,)), workspace.numel(),
                 _stream(stream)), "s2_pipeline_dense_host")


# ---- allocation helpers (torch owns the memory; the library never allocates) ----

def alloc_encode_outputs(W: int, n: int, d: int, w: int, device="cuda") -> Tuple[torch.Tensor, torch.Tensor]:
    return (torch.empty((W, nwords(n)), dtype=torch.int32, device=device),
            torch.empty((W, d, w), dtype=torch.float32, device=device))

