"""ctypes binding of libexl3.so (argument marshalling only).

Every function takes torch tensors that already live on the GPU, checks
dtype/contiguity/device, and passes raw pointers, sizes and the current CUDA
stream to the C ABI.  All arithmetic happens in the library's kernels.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libexl3.so")
_lib: Optional[ctypes.CDLL] = None

CODEBOOKS = {"3inst": 0, "mcg": 1, "mul1": 2}
_F16, _BF16 = 0, 1
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "split-k workspace too small", 4: "CUDA error"}


class Exl3Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = ""
        if status == 4 and _lib is not None:
            detail = ": " + _lib.exl3_last_error().decode()
        super().__init__(f"{what} failed: {_STATUS.get(status, status)}{detail}")


def lib() -> ctypes.CDLL:
    """Load libexl3.so (built in-tree by ``build_ext.build()``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)"
        )
    L = ctypes.CDLL(_LIB_PATH)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    L.exl3_input_transform.argtypes = [vp, ctypes.c_int, i64, i64, vp, i32, vp, vp]
    L.exl3_moe_input_transform.argtypes = [vp, ctypes.c_int, i64, i64, vp, i64, i32, vp, i32, vp, i32, i32, vp, vp]
    L.exl3_moe_input_transform.restype = ctypes.c_int
    L.exl3_moe_gemm.argtypes = [vp, i64, i64, vp, i32, ctypes.c_int, vp, vp, i32, vp, i32, i32, vp, ctypes.c_int,
                                i64, vp]
    L.exl3_moe_gemm.restype = ctypes.c_int
    L.exl3_moe_combine.argtypes = [vp, ctypes.c_int, i64, i64, vp, vp, i32, i32, vp, i64, i32, vp, vp, ctypes.c_int, vp]
    L.exl3_moe_combine.restype = ctypes.c_int
    L.exl3_input_transform_swiglu.argtypes = [vp, ctypes.c_int, i64, i64, vp, i32, vp, vp]
    L.exl3_input_transform_swiglu.restype = ctypes.c_int
    L.exl3_gemm.argtypes = [vp, i64, i64, vp, i32, ctypes.c_int, vp, vp, i32, vp, ctypes.c_int, i64, vp]
    L.exl3_gemm_splitk.argtypes = L.exl3_gemm.argtypes[:-1] + [vp, sz, vp]
    L.exl3_gemm_splitk_noalloc.argtypes = L.exl3_gemm.argtypes
    L.exl3_gemm_splitk_noalloc.restype = ctypes.c_int
    L.exl3_splitk_parts.argtypes = [i64, i64]
    L.exl3_splitk_parts.restype = i32
    L.exl3_splitk_workspace_bytes.argtypes = [i64, i64, i64]
    L.exl3_splitk_workspace_bytes.restype = sz
    L.exl3_test_gemm_shape.argtypes = [i32] + L.exl3_gemm.argtypes[:-1] + [vp, sz, vp]
    L.exl3_test_gemm_shape.restype = ctypes.c_int
    L.exl3_test_codebook.argtypes = [ctypes.c_int, vp, vp]
    L.exl3_test_unpack.argtypes = [vp, i32, ctypes.c_int, i64, i64, vp, vp]
    L.exl3_test_tile_plan.argtypes = [i64, i64, i64, ctypes.POINTER(ctypes.c_int32), i32, i32,
                                      ctypes.POINTER(ctypes.c_int64)]
    L.exl3_test_tile_plan.restype = ctypes.c_int
    L.exl3_test_wait_timeout.argtypes = [vp, vp]
    L.exl3_test_wait_timeout.restype = ctypes.c_int
    L.exl3_set_autotune.argtypes = [i32]
    L.exl3_set_autotune.restype = ctypes.c_int
    L.exl3_clear_autotune.argtypes = []
    L.exl3_clear_autotune.restype = ctypes.c_int
    L.exl3_autotune_entries.argtypes = []
    L.exl3_autotune_entries.restype = i64
    L.exl3_status_string.argtypes = [ctypes.c_int]
    L.exl3_status_string.restype = ctypes.c_char_p
    L.exl3_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    L.exl3_device_status.restype = ctypes.c_int
    L.exl3_last_error.argtypes = []
    L.exl3_last_error.restype = ctypes.c_char_p
    for name in ("exl3_input_transform", "exl3_gemm", "exl3_gemm_splitk", "exl3_test_codebook", "exl3_test_unpack"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def device_status() -> int:
    """Read and clear the kernels' device-side error flags (synchronises the device)."""
    flags = ctypes.c_uint32(0)
    _check(lib().exl3_device_status(ctypes.byref(flags)), "exl3_device_status")
    return int(flags.value)


def test_wait_timeout(device="cuda") -> int:
    """exl3_test_wait_timeout: a kernel whose bounded wait gives up (about 2 s);
    returns the kernel's out word (0 when the wait gave up)."""
    out = torch.full((1,), 7, dtype=torch.int32, device=device)
    _check(lib().exl3_test_wait_timeout(_ptr(out), _stream(out)), "exl3_test_wait_timeout")
    return int(out.item())


def test_tile_plan(m: int, k: int, n: int, shard_cols: Sequence[int], split: bool = False) -> tuple:
    """The cost model's plan (host only): (shape, tail shape or -1, pair tiles, tail row, tail column)."""
    cols, ns = _cols(shard_cols)
    out = (ctypes.c_int64 * 5)()
    _check(lib().exl3_test_tile_plan(m, k, n, cols, ns, 1 if split else 0, out), "exl3_test_tile_plan")
    return tuple(int(v) for v in out)


def set_autotune(enable: bool) -> None:
    """Tile-shape autotune: time every shape on a key's first uncaptured call and keep the fastest."""
    _check(lib().exl3_set_autotune(1 if enable else 0), "exl3_set_autotune")


def clear_autotune() -> None:
    _check(lib().exl3_clear_autotune(), "exl3_clear_autotune")


def autotune_entries() -> int:
    return int(lib().exl3_autotune_entries())


def status_string(status: int) -> str:
    return lib().exl3_status_string(status).decode()


def _check(status: int, what: str) -> None:
    if status != 0:
        raise Exl3Error(status, what)


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, dtype, name: str) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _cols(shard_cols: Sequence[int]):
    arr = (ctypes.c_int32 * len(shard_cols))(*[int(c) for c in shard_cols])
    return arr, len(shard_cols) - 1


def splitk_parts(k: int, n: int) -> int:
    return int(lib().exl3_splitk_parts(k, n))


def splitk_workspace_bytes(m: int, k: int, n: int) -> int:
    return int(lib().exl3_splitk_workspace_bytes(m, k, n))


def input_transform(x: torch.Tensor, suh: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """xh[s] = fp16(H(x * suh[s]) * 2^-4) for every shard; x bf16/fp16 [m, k], suh fp16 [S, k]."""
    if x.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("x must be bf16 or fp16")
    _need(x, x.dtype, "x")
    _need(suh, torch.float16, "suh")
    m, k = x.shape
    s = suh.shape[0]
    if out is None:
        out = torch.empty((s, m, k), dtype=torch.float16, device=x.device)
    _need(out, torch.float16, "out")
    st = lib().exl3_input_transform(_ptr(x), _BF16 if x.dtype == torch.bfloat16 else _F16, m, k, _ptr(suh), s,
                                    _ptr(out), _stream(x))
    _check(st, "exl3_input_transform")
    return out


def input_transform_swiglu(gate_up: torch.Tensor, suh: torch.Tensor,
                           out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """xh[s] = fp16(H(silu(gate) * up * suh[s]) * 2^-4); gate_up bf16/fp16 [m, 2k] (gate first), suh fp16 [S, k]."""
    if gate_up.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("gate_up must be bf16 or fp16")
    _need(gate_up, gate_up.dtype, "gate_up")
    _need(suh, torch.float16, "suh")
    m, k2 = gate_up.shape
    if k2 % 2:
        raise ValueError("gate_up holds gate and up halves")
    k = k2 // 2
    s = suh.shape[0]
    if out is None:
        out = torch.empty((s, m, k), dtype=torch.float16, device=gate_up.device)
    _need(out, torch.float16, "out")
    st = lib().exl3_input_transform_swiglu(_ptr(gate_up), _BF16 if gate_up.dtype == torch.bfloat16 else _F16, m, k,
                                           _ptr(suh), s, _ptr(out), _stream(gate_up))
    _check(st, "exl3_input_transform_swiglu")
    return out


def moe_input_transform(x: torch.Tensor, sorted_ids: torch.Tensor, topk: int, block_expert: torch.Tensor,
                        block: int, suh: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Gather and rotate block-aligned routed rows; suh fp16 [E, S, k] -> xh fp16 [S, rows, k]."""
    if x.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("x must be bf16 or fp16")
    _need(x, x.dtype, "x")
    _need(sorted_ids, torch.int32, "sorted_ids")
    _need(block_expert, torch.int32, "block_expert")
    _need(suh, torch.float16, "suh")
    num_tokens, k = x.shape
    e, s, _ = suh.shape
    rows = sorted_ids.numel()
    if out is None:
        out = torch.empty((s, rows, k), dtype=torch.float16, device=x.device)
    _need(out, torch.float16, "out")
    st = lib().exl3_moe_input_transform(_ptr(x), _BF16 if x.dtype == torch.bfloat16 else _F16, num_tokens, k,
                                        _ptr(sorted_ids), rows, int(topk), _ptr(block_expert), int(block), _ptr(suh),
                                        s, e, _ptr(out), _stream(x))
    _check(st, "exl3_moe_input_transform")
    return out


def moe_gemm(xh: torch.Tensor, trellis: torch.Tensor, bits: int, cb, svh: torch.Tensor, shard_cols: Sequence[int],
             block_expert: torch.Tensor, block: int, out_dtype=torch.bfloat16,
             out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Grouped GEMM; trellis int16 [E, k/16, n/16, 16*bits], svh fp16 [E, n] -> y [rows, n] (padded-row order)."""
    _need(xh, torch.float16, "xh")
    _need(trellis, torch.int16, "trellis")
    _need(svh, torch.float16, "svh")
    _need(block_expert, torch.int32, "block_expert")
    s, rows, k = xh.shape
    e, n = svh.shape
    if out is None:
        out = torch.empty((rows, n), dtype=out_dtype, device=xh.device)
    if out.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("output must be bf16 or fp16")
    _need(out, out.dtype, "out")
    cols, ns = _cols(shard_cols)
    cbid = CODEBOOKS[cb] if isinstance(cb, str) else int(cb)
    st = lib().exl3_moe_gemm(_ptr(xh), rows, k, _ptr(trellis), bits, cbid, _ptr(svh), cols, ns, _ptr(block_expert),
                             int(block), e, _ptr(out), _BF16 if out.dtype == torch.bfloat16 else _F16, n, _stream(xh))
    _check(st, "exl3_moe_gemm")
    return out


def moe_combine(y: torch.Tensor, sorted_ids: torch.Tensor, block_expert: torch.Tensor, block: int,
                num_experts: int, weights: torch.Tensor, topk: int, out_dtype=torch.bfloat16,
                out: Optional[torch.Tensor] = None, pair_rows: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Weighted sum of each token's top-k rows of a grouped GEMM's output:
    y [rows, n] (bf16/fp16), weights fp32 [tokens, topk] -> out [tokens, n].
    pair_rows is int32 [tokens * topk] scratch (allocated when not given)."""
    if y.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("y must be bf16 or fp16")
    _need(y, y.dtype, "y")
    _need(sorted_ids, torch.int32, "sorted_ids")
    _need(block_expert, torch.int32, "block_expert")
    _need(weights, torch.float32, "weights")
    rows, n = y.shape
    num_tokens = weights.shape[0]
    if weights.shape != (num_tokens, topk):
        raise ValueError("weights must be [tokens, topk]")
    if out is None:
        out = torch.empty((num_tokens, n), dtype=out_dtype, device=y.device)
    if out.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("output must be bf16 or fp16")
    _need(out, out.dtype, "out")
    if pair_rows is None:
        pair_rows = torch.empty(max(1, num_tokens * topk), dtype=torch.int32, device=y.device)
    _need(pair_rows, torch.int32, "pair_rows")
    st = lib().exl3_moe_combine(_ptr(y), _BF16 if y.dtype == torch.bfloat16 else _F16, rows, n, _ptr(sorted_ids),
                                _ptr(block_expert), int(block), int(num_experts), _ptr(weights), num_tokens,
                                int(topk), _ptr(pair_rows), _ptr(out), _BF16 if out.dtype == torch.bfloat16 else _F16,
                                _stream(y))
    _check(st, "exl3_moe_combine")
    return out


def _gemm_common(xh, trellis, bits, cb, svh, shard_cols, out_dtype, out):
    _need(xh, torch.float16, "xh")
    _need(trellis, torch.int16, "trellis")
    _need(svh, torch.float16, "svh")
    s, m, k = xh.shape
    n = int(shard_cols[-1])
    if out is None:
        out = torch.empty((m, n), dtype=out_dtype, device=xh.device)
    if out.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("output must be bf16 or fp16")
    _need(out, out.dtype, "out")
    cols, ns = _cols(shard_cols)
    if ns != s:
        raise ValueError("xh holds one slice per shard")
    cbid = CODEBOOKS[cb] if isinstance(cb, str) else int(cb)
    return m, k, n, cols, ns, cbid, out


def gemm(xh: torch.Tensor, trellis: torch.Tensor, bits: int, cb, svh: torch.Tensor, shard_cols: Sequence[int],
         out_dtype=torch.bfloat16, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    m, k, n, cols, ns, cbid, out = _gemm_common(xh, trellis, bits, cb, svh, shard_cols, out_dtype, out)
    st = lib().exl3_gemm(_ptr(xh), m, k, _ptr(trellis), bits, cbid, _ptr(svh), cols, ns, _ptr(out),
                         _BF16 if out.dtype == torch.bfloat16 else _F16, n, _stream(xh))
    _check(st, "exl3_gemm")
    return out


def gemm_splitk(xh: torch.Tensor, trellis: torch.Tensor, bits: int, cb, svh: torch.Tensor,
                shard_cols: Sequence[int], acc: torch.Tensor, out_dtype=torch.bfloat16,
                out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Split-k variant; ``acc`` is an fp32 workspace of at least splitk_workspace_bytes (any contents;
    the call leaves it zeroed)."""
    m, k, n, cols, ns, cbid, out = _gemm_common(xh, trellis, bits, cb, svh, shard_cols, out_dtype, out)
    _need(acc, torch.float32, "acc")
    st = lib().exl3_gemm_splitk(_ptr(xh), m, k, _ptr(trellis), bits, cbid, _ptr(svh), cols, ns, _ptr(out),
                                _BF16 if out.dtype == torch.bfloat16 else _F16, n, _ptr(acc),
                                acc.numel() * 4, _stream(xh))
    _check(st, "exl3_gemm_splitk")
    return out


# Size of the library's built-in split-k scratch (EXL3_NOALLOC_SCRATCH_BYTES in include/exl3.h).
NOALLOC_SCRATCH_BYTES = 8 << 20


def gemm_splitk_noalloc(xh: torch.Tensor, trellis: torch.Tensor, bits: int, cb, svh: torch.Tensor,
                        shard_cols: Sequence[int], out_dtype=torch.bfloat16,
                        out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Split-k GEMM whose partials live in the library's built-in scratch array.

    For callers that cannot allocate a workspace.  Requests whose workspace
    would exceed NOALLOC_SCRATCH_BYTES are refused; calls must not overlap on
    the GPU (they share the one array).
    """
    m, k, n, cols, ns, cbid, out = _gemm_common(xh, trellis, bits, cb, svh, shard_cols, out_dtype, out)
    st = lib().exl3_gemm_splitk_noalloc(_ptr(xh), m, k, _ptr(trellis), bits, cbid, _ptr(svh), cols, ns, _ptr(out),
                                        _BF16 if out.dtype == torch.bfloat16 else _F16, n, _stream(xh))
    if st == 3:
        raise Exl3Error(st, f"exl3_gemm_splitk_noalloc (needs {splitk_workspace_bytes(m, k, n)} bytes of scratch, "
                            f"the built-in array holds {NOALLOC_SCRATCH_BYTES})")
    _check(st, "exl3_gemm_splitk_noalloc")
    return out


def linear(x: torch.Tensor, trellis: torch.Tensor, bits: int, cb, suh: torch.Tensor, svh: torch.Tensor,
           shard_cols: Sequence[int], out_dtype=torch.bfloat16, acc: Optional[torch.Tensor] = None,
           xh: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Whole layer: input rotation, then the GEMM (split-k when ``acc`` is given)."""
    xh = input_transform(x, suh, xh)
    if acc is not None:
        return gemm_splitk(xh, trellis, bits, cb, svh, shard_cols, acc, out_dtype, out)
    return gemm(xh, trellis, bits, cb, svh, shard_cols, out_dtype, out)


# Tile shapes exl3_test_gemm_shape accepts (EXL3_TEST_TILE_SHAPES in include/exl3.h).
TEST_TILE_SHAPES = 29


def test_gemm_shape(tile_shape: int, xh: torch.Tensor, trellis: torch.Tensor, bits: int, cb, svh: torch.Tensor,
                    shard_cols: Sequence[int], acc: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16,
                    out: Optional[torch.Tensor] = None) -> Optional[torch.Tensor]:
    """exl3_gemm (or the split-k GEMM when ``acc`` is given) with a fixed tile shape.

    Returns None, launching nothing, when the shape cannot run the call.
    """
    m, k, n, cols, ns, cbid, out = _gemm_common(xh, trellis, bits, cb, svh, shard_cols, out_dtype, out)
    if acc is not None:
        _need(acc, torch.float32, "acc")
    st = lib().exl3_test_gemm_shape(int(tile_shape), _ptr(xh), m, k, _ptr(trellis), bits, cbid, _ptr(svh), cols, ns,
                                    _ptr(out), _BF16 if out.dtype == torch.bfloat16 else _F16, n,
                                    _ptr(acc) if acc is not None else None, acc.numel() * 4 if acc is not None else 0,
                                    _stream(xh))
    if st == 2:
        return None
    _check(st, "exl3_test_gemm_shape")
    return out


def test_codebook(cb, device="cuda") -> torch.Tensor:
    """fp16 bit patterns (as int16) of the codebook at all 65,536 states."""
    out = torch.empty(65536, dtype=torch.int16, device=device)
    cbid = CODEBOOKS[cb] if isinstance(cb, str) else int(cb)
    _check(lib().exl3_test_codebook(cbid, _ptr(out), _stream(out)), "exl3_test_codebook")
    return out


def test_unpack(trellis: torch.Tensor, bits: int, cb) -> torch.Tensor:
    """Dense Wq [k, n] (fp16 bit patterns as int16) decoded by the library."""
    _need(trellis, torch.int16, "trellis")
    kt, nt, w = trellis.shape
    if w != 16 * bits:
        raise ValueError("trellis last axis must be 16*bits")
    out = torch.empty((16 * kt, 16 * nt), dtype=torch.int16, device=trellis.device)
    cbid = CODEBOOKS[cb] if isinstance(cb, str) else int(cb)
    st = lib().exl3_test_unpack(_ptr(trellis), bits, cbid, 16 * kt, 16 * nt, _ptr(out), _stream(trellis))
    _check(st, "exl3_test_unpack")
    return out
