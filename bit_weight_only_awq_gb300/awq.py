"""ctypes binding over libawq.so (declared in include/awq.h), same entry-point names.

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels.  PyTorch provides device memory (outputs and workspaces allocated
here when the caller passes none) and the current CUDA stream.  Importing this
module loads the library and raises ImportError when it has not been built;
there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os
import re

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libawq.so")
_HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "awq.h")

if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing: build it with `python -m bit_weight_only_awq_gb300.build`")
lib = ctypes.CDLL(_LIB_PATH)

STATUS = {0: "AWQ_OK", -1: "AWQ_EINVAL", -2: "AWQ_EALIGN", -3: "AWQ_EARCH", -4: "AWQ_ECUDA",
          -5: "AWQ_ETIMEOUT", -6: "AWQ_EWORKSPACE", -7: "AWQ_ENULL"}
OP_GEMV, OP_GEMM, OP_W4A8_GEMM, OP_GEMV_PREPACKED, OP_GEMV_BF16, OP_GEMM_BF16, OP_W4A8_GROUPED = 0, 1, 2, 3, 4, 5, 6
GROUP_SIZE = 128

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t

_SIGS = {
    "awq_status_string": (ctypes.c_char_p, [_i32]),
    "awq_pack": (_i32, [_p, _i64, _i64, _p, _p]),
    "awq_unpack": (_i32, [_p, _i64, _i64, _p, _p]),
    "awq_pack_order": (_i32, [_p, _i64, _i64, _i32, _p, _p]),
    "awq_unpack_order": (_i32, [_p, _i64, _i64, _i32, _p, _p]),
    "awq_dequant": (_i32, [_p, _p, _p, _i64, _i64, _i32, _p, _p]),
    "awq_workspace_bytes": (_sz, [_i32, _i64, _i64, _i64, _i32]),
    "awq_gemv": (_i32, [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i32, _i32, _p, _sz, _p]),
    "awq_gemm": (_i32, [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i32, _i32, _p, _sz, _p]),
    "awq_gemv_noalloc": (_i32, [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i32, _i32, _p]),
    "w4a8_quant_act": (_i32, [_p, _p, _p, _i64, _i64, _p]),
    "w4a8_gemm": (_i32, [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i32, _p, _sz, _p]),
    "w4a8_linear": (_i32, [_p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i32, _p, _sz, _p]),
    "awq_dequant_bf16": (_i32, [_p, _p, _p, _i64, _i64, _i32, _p, _p]),
    "awq_gemv_bf16": (_i32, [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i32, _i32, _p, _sz, _p]),
    "awq_gemm_bf16": (_i32, [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i32, _i32, _p, _sz, _p]),
    "awq_prepacked_bytes": (_sz, [_i64, _i64]),
    "awq_prepack_gemv": (_i32, [_p, _p, _p, _i64, _i64, _i32, _p, _sz, _p]),
    "awq_unprepack_gemv": (_i32, [_p, _i64, _i64, _p, _p, _p, _p]),
    "awq_gemv_prepacked": (_i32, [_p, _p, _p, _i64, _i64, _i64, _i32, _p, _sz, _p]),
    "w4a8_gemm_grouped": (_i32, [_p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i32, _i32, _p, _sz, _p]),
    "w4a8_linear_grouped": (_i32, [_p, _p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i32, _i32, _p, _sz, _p]),
    "awq_last_device_error": (_i32, [ctypes.POINTER(_i32)]),
    "awq_selftest_wait_timeout": (_i32, [_i64, _p]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


def header_functions() -> list[str]:
    """Names of the functions declared in include/awq.h."""
    with open(_HEADER) as fh:
        text = fh.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*((?:awq|w4a8)_[a-z0-9_]+)\s*\(", text, re.M)))


class AwqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = lib.awq_status_string(status).decode()
        super().__init__(f"{fn}: {msg}")
        self.status = status


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise AwqError(fn, status)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


# One zero-filled workspace per device, grown on demand.  The library leaves its tile
# counters at zero after every call, so reuse on one stream needs no re-zeroing.
_workspaces: dict[int, torch.Tensor] = {}


def device_workspace(nbytes: int, device: torch.device) -> torch.Tensor | None:
    if nbytes == 0:
        return None
    idx = device.index if device.index is not None else torch.cuda.current_device()
    ws = _workspaces.get(idx)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _workspaces[idx] = ws
    return ws


def awq_workspace_bytes(op: int, M: int, K: int, N: int, split_k: int = 0) -> int:
    return int(lib.awq_workspace_bytes(op, M, K, N, split_k))


# Workspace sizes by (op, M, K, N, split_k, device): the size depends only on these (the plan reads
# the device's SM count), and a decode loop repeats the same few shapes.
_ws_need: dict[tuple, int] = {}


def _workspace_need(op: int, M: int, K: int, N: int, split_k: int, device: torch.device) -> int:
    key = (op, M, K, N, split_k, device.index)
    need = _ws_need.get(key)
    if need is None:
        need = _ws_need[key] = awq_workspace_bytes(op, M, K, N, split_k)
    return need


def awq_pack(q: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    rows, n = q.shape
    if out is None:
        out = torch.empty((rows, n // 8), dtype=torch.int32, device=q.device)
    _check("awq_pack", lib.awq_pack(_ptr(q), rows, n, _ptr(out), _stream(stream)))
    return out


def awq_unpack(packed: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    rows, nw = packed.shape
    if out is None:
        out = torch.empty((rows, nw * 8), dtype=torch.uint8, device=packed.device)
    _check("awq_unpack", lib.awq_unpack(_ptr(packed), rows, nw * 8, _ptr(out), _stream(stream)))
    return out


ORDER_OLD, ORDER_NEW = 0, 1


def awq_pack_order(q: torch.Tensor, order: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    rows, n = q.shape
    if out is None:
        out = torch.empty((rows, n // 8), dtype=torch.int32, device=q.device)
    _check("awq_pack_order", lib.awq_pack_order(_ptr(q), rows, n, order, _ptr(out), _stream(stream)))
    return out


def awq_unpack_order(packed: torch.Tensor, order: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    rows, nw = packed.shape
    if out is None:
        out = torch.empty((rows, nw * 8), dtype=torch.uint8, device=packed.device)
    _check("awq_unpack_order", lib.awq_unpack_order(_ptr(packed), rows, nw * 8, order, _ptr(out), _stream(stream)))
    return out


def awq_dequant(qweight, qzeros, scales, group_size: int = GROUP_SIZE, out=None, stream=None) -> torch.Tensor:
    K, nw = qweight.shape
    if out is None:
        out = torch.empty((K, nw * 8), dtype=torch.float16, device=qweight.device)
    _check("awq_dequant", lib.awq_dequant(_ptr(qweight), _ptr(qzeros), _ptr(scales), K, nw * 8, group_size,
                                          _ptr(out), _stream(stream)))
    return out


def _gemm_like(name, op, x, qweight, qzeros, scales, group_size, split_k, out, ws, stream):
    M, K = x.shape
    N = qweight.shape[1] * 8
    if out is None:
        out = torch.empty((M, N), dtype=x.dtype, device=x.device)
    if ws is None:
        ws = device_workspace(_workspace_need(op, M, K, N, split_k, x.device), x.device)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    fn = getattr(lib, name)
    _check(name, fn(_ptr(x), _ptr(qweight), _ptr(qzeros), _ptr(scales), _ptr(out), M, K, N, group_size,
                    split_k, _ptr(ws), nbytes, _stream(stream)))
    return out


def awq_gemv(x, qweight, qzeros, scales, group_size: int = GROUP_SIZE, split_k: int = 0, out=None,
             workspace=None, stream=None) -> torch.Tensor:
    return _gemm_like("awq_gemv", OP_GEMV, x, qweight, qzeros, scales, group_size, split_k, out, workspace, stream)


def awq_gemv_noalloc(x, qweight, qzeros, scales, group_size: int = GROUP_SIZE, split_k: int = 0, out=None,
                     stream=None) -> torch.Tensor:
    """awq_gemv without a caller workspace: the library's fixed per-device scratch array is used.

    The output tensor is the only memory this wrapper allocates (pass `out` to allocate nothing).
    """
    M, K = x.shape
    N = qweight.shape[1] * 8
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _check("awq_gemv_noalloc", lib.awq_gemv_noalloc(_ptr(x), _ptr(qweight), _ptr(qzeros), _ptr(scales), _ptr(out),
                                                    M, K, N, group_size, split_k, _stream(stream)))
    return out


class Prepacked:
    """A prepared decode copy of an AWQ layer (awq_prepack_gemv): the device bytes and the shape."""

    def __init__(self, data: torch.Tensor, K: int, N: int):
        self.data, self.K, self.N = data, K, N


def awq_prepack_gemv(qweight, qzeros, scales, group_size: int = GROUP_SIZE, stream=None) -> Prepacked:
    K, nw = qweight.shape
    N = nw * 8
    nbytes = int(lib.awq_prepacked_bytes(K, N))
    if nbytes == 0:
        raise AwqError("awq_prepack_gemv", -1)
    data = torch.empty(nbytes, dtype=torch.uint8, device=qweight.device)
    _check("awq_prepack_gemv", lib.awq_prepack_gemv(_ptr(qweight), _ptr(qzeros), _ptr(scales), K, N, group_size,
                                                    _ptr(data), nbytes, _stream(stream)))
    return Prepacked(data, K, N)


def awq_unprepack_gemv(packed: Prepacked, with_zeros: bool = True, stream=None):
    """The AWQ (qweight, qzeros or None, scales) that `packed` was made from."""
    K, N = packed.K, packed.N
    dev = packed.data.device
    qweight = torch.empty((K, N // 8), dtype=torch.int32, device=dev)
    qzeros = torch.empty((K // GROUP_SIZE, N // 8), dtype=torch.int32, device=dev) if with_zeros else None
    scales = torch.empty((K // GROUP_SIZE, N), dtype=torch.float16, device=dev)
    _check("awq_unprepack_gemv", lib.awq_unprepack_gemv(_ptr(packed.data), K, N, _ptr(qweight), _ptr(qzeros),
                                                        _ptr(scales), _stream(stream)))
    return qweight, qzeros, scales


def awq_gemv_prepacked(x, packed: Prepacked, split_k: int = 0, out=None, workspace=None, stream=None):
    M, K = x.shape
    N = packed.N
    if K != packed.K:
        raise ValueError("x has K columns different from the prepared layer's")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    ws = workspace if workspace is not None else \
        device_workspace(_workspace_need(OP_GEMV_PREPACKED, M, K, N, split_k, x.device), x.device)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check("awq_gemv_prepacked", lib.awq_gemv_prepacked(_ptr(x), _ptr(packed.data), _ptr(out), M, K, N, split_k,
                                                        _ptr(ws), nbytes, _stream(stream)))
    return out


def awq_gemm(x, qweight, qzeros, scales, group_size: int = GROUP_SIZE, split_k: int = 0, out=None,
             workspace=None, stream=None) -> torch.Tensor:
    return _gemm_like("awq_gemm", OP_GEMM, x, qweight, qzeros, scales, group_size, split_k, out, workspace, stream)


def _need_bf16(*tensors):
    for t in tensors:
        if t is not None and t.dtype != torch.bfloat16:
            raise TypeError("the bf16 entry points take bf16 activations and scales")


def awq_dequant_bf16(qweight, qzeros, scales, group_size: int = GROUP_SIZE, out=None, stream=None):
    _need_bf16(scales)
    K, nw = qweight.shape
    if out is None:
        out = torch.empty((K, nw * 8), dtype=torch.bfloat16, device=qweight.device)
    _check("awq_dequant_bf16", lib.awq_dequant_bf16(_ptr(qweight), _ptr(qzeros), _ptr(scales), K, nw * 8,
                                                    group_size, _ptr(out), _stream(stream)))
    return out


def awq_gemv_bf16(x, qweight, qzeros, scales, group_size: int = GROUP_SIZE, split_k: int = 0, out=None,
                  workspace=None, stream=None) -> torch.Tensor:
    _need_bf16(x, scales)
    return _gemm_like("awq_gemv_bf16", OP_GEMV_BF16, x, qweight, qzeros, scales, group_size, split_k, out,
                      workspace, stream)


def awq_gemm_bf16(x, qweight, qzeros, scales, group_size: int = GROUP_SIZE, split_k: int = 0, out=None,
                  workspace=None, stream=None) -> torch.Tensor:
    _need_bf16(x, scales)
    return _gemm_like("awq_gemm_bf16", OP_GEMM_BF16, x, qweight, qzeros, scales, group_size, split_k, out,
                      workspace, stream)


GEMV_MAX_M = 16


def awq_linear(x, qweight, qzeros, scales, group_size: int = GROUP_SIZE, **kw) -> torch.Tensor:
    """The pages' dispatch by token count, with the threshold moved from 8 to 16: the GEMV kernel
    streams the weights once for up to 16 tokens (two 8-token halves) and was measured 1.3-2.9x
    faster than the tensor-core GEMM at 16 tokens; the GEMM above."""
    fn = awq_gemv if x.shape[0] <= GEMV_MAX_M else awq_gemm
    return fn(x, qweight, qzeros, scales, group_size, **kw)


def w4a8_quant_act(x, xq=None, s_tok=None, stream=None):
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if s_tok is None:
        s_tok = torch.empty((M,), dtype=torch.float32, device=x.device)
    _check("w4a8_quant_act", lib.w4a8_quant_act(_ptr(x), _ptr(xq), _ptr(s_tok), M, K, _stream(stream)))
    return xq, s_tok


def w4a8_gemm(xq, s_tok, wq, s_ch, split_k: int = 0, out=None, acc_out=None, workspace=None, stream=None):
    M, K = xq.shape
    N = wq.shape[1] * 8
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=xq.device)
    need = awq_workspace_bytes(OP_W4A8_GEMM, M, K, N, split_k)
    ws = workspace if workspace is not None else device_workspace(need, xq.device)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check("w4a8_gemm", lib.w4a8_gemm(_ptr(xq), _ptr(s_tok), _ptr(wq), _ptr(s_ch), _ptr(out), _ptr(acc_out), M, K,
                                      N, split_k, _ptr(ws), nbytes, _stream(stream)))
    return out


def w4a8_linear(x, wq, s_ch, split_k: int = 0, out=None, acc_out=None, xq_out=None, s_tok=None, workspace=None,
                stream=None):
    """W4A8 from fp16 activations in one call (quantization fused); returns (y, s_tok)."""
    M, K = x.shape
    N = wq.shape[1] * 8
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    if s_tok is None:
        s_tok = torch.empty((M,), dtype=torch.float32, device=x.device)
    need = awq_workspace_bytes(OP_W4A8_GEMM, M, K, N, split_k)
    ws = workspace if workspace is not None else device_workspace(need, x.device)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check("w4a8_linear", lib.w4a8_linear(_ptr(x), _ptr(wq), _ptr(s_ch), _ptr(out), _ptr(acc_out), _ptr(xq_out),
                                          _ptr(s_tok), M, K, N, split_k, _ptr(ws), nbytes, _stream(stream)))
    return out, s_tok


def w4a8_gemm_grouped(xq, s_tok, wq, s3, s2, split_k: int = 0, out=None, acc_out=None, workspace=None,
                      stream=None):
    """Per-group W4A8 from int8 codes (s3: integer group factors 1..16, s2: channel scales)."""
    M, K = xq.shape
    N = wq.shape[1] * 8
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=xq.device)
    need = awq_workspace_bytes(OP_W4A8_GROUPED, M, K, N, split_k)
    ws = workspace if workspace is not None else device_workspace(need, xq.device)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check("w4a8_gemm_grouped", lib.w4a8_gemm_grouped(_ptr(xq), _ptr(s_tok), _ptr(wq), _ptr(s3), _ptr(s2), _ptr(out),
                                                      _ptr(acc_out), M, K, N, GROUP_SIZE, split_k, _ptr(ws), nbytes,
                                                      _stream(stream)))
    return out


def w4a8_linear_grouped(x, wq, s3, s2, split_k: int = 0, out=None, acc_out=None, xq_out=None, s_tok=None,
                        workspace=None, stream=None):
    """Per-group W4A8 from fp16 activations in one call (quantization included); returns (y, s_tok)."""
    M, K = x.shape
    N = wq.shape[1] * 8
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    if s_tok is None:
        s_tok = torch.empty((M,), dtype=torch.float32, device=x.device)
    need = awq_workspace_bytes(OP_W4A8_GROUPED, M, K, N, split_k)
    ws = workspace if workspace is not None else device_workspace(need, x.device)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check("w4a8_linear_grouped", lib.w4a8_linear_grouped(_ptr(x), _ptr(wq), _ptr(s3), _ptr(s2), _ptr(out),
                                                          _ptr(acc_out), _ptr(xq_out), _ptr(s_tok), M, K, N,
                                                          GROUP_SIZE, split_k, _ptr(ws), nbytes, _stream(stream)))
    return out, s_tok


def awq_last_device_error() -> int:
    code = _i32(0)
    status = lib.awq_last_device_error(ctypes.byref(code))
    if status not in (0, -5):
        raise AwqError("awq_last_device_error", status)
    return int(code.value)


def awq_selftest_wait_timeout(limit_ns: int = 1_000_000, stream=None) -> None:
    """Run one bounded device wait that expires after `limit_ns` (see include/awq.h)."""
    _check("awq_selftest_wait_timeout", lib.awq_selftest_wait_timeout(int(limit_ns), _stream(stream)))
