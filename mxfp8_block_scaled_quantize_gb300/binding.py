"""ctypes binding to libtemx.so (argument marshalling only).

The ``te_mx_*`` functions take raw integer pointers and mirror include/temx.h;
they raise ``TemxError`` on any status other than TE_MX_OK.  The torch-level
helpers (``quantize``, ``gemm``, ``grouped_gemm``) only allocate outputs with
torch and pass ``data_ptr()`` and the current stream; every step of the
computation runs in the library's CUDA kernels.  There is no fallback: if the
library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libtemx.so")

TE_MX_OK = 0
STATUS_NAMES = {0: "TE_MX_OK", 1: "TE_MX_ERR_INVALID_ARG", 2: "TE_MX_ERR_UNSUPPORTED_SHAPE",
                3: "TE_MX_ERR_MISALIGNED", 4: "TE_MX_ERR_WORKSPACE_TOO_SMALL", 5: "TE_MX_ERR_CUDA",
                6: "TE_MX_ERR_DEVICE_TIMEOUT", 7: "TE_MX_ERR_ARCH"}
EPI_NONE, EPI_BIAS, EPI_GELU_AUX, EPI_BIAS_GELU_AUX, EPI_DGELU, EPI_ACCUMULATE_F32 = 0, 1, 2, 3, 4, 5

# (name, restype, argtypes) for every function declared in include/temx.h
_I64, _I32, _P, _SZ = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
SIGNATURES = {
    "te_mx_scale_pitch": (_SZ, [_I64]),
    "te_mx_quantize": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _I64, _P, _P, _I64, _P]),
    "te_mx_block_quantize": (ctypes.c_int, [_P, _I64, _I64, _I64, _I32, _P, _P, _I64, _P, _P, _I64, _P]),
    "te_mx_block_scale_pitch_fp32": (_I64, [_I64]),
    "te_mx_block_quantize_fp32": (ctypes.c_int, [_P, _I64, _I64, _I64, _I32, _P, _P, _I64, _P, _P, _I64, _P]),
    "te_mx_layernorm_quantize": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, ctypes.c_float, _P, _P, _I64, _P,
                                                _P, _I64, _P, _P, _P]),
    "te_mx_grouped_code_width": (_I64, [_I64, _I32]),
    "te_mx_grouped_scale_width": (_I64, [_I64, _I32]),
    "te_mx_quantize_colwise_grouped": (ctypes.c_int, [_P, _I64, _I64, _I64, _I32, _P, _P, _I64, _P, _I64, _P]),
    "te_mx_grouped_gemm_wgrad": (ctypes.c_int, [_I32, _P, _I64, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I32, _P,
                                                _P]),
    "te_mx_quantize_dbias_workspace_size": (_SZ, [_I64, _I64]),
    "te_mx_quantize_dbias": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _I64, _P, _P, _I64, _P, _P, _SZ, _P]),
    "te_mx_quantize_dbias_noalloc": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _I64, _P, _P, _I64, _P, _P]),
    "te_mx_gemm": (ctypes.c_int, [_P, _P, _I64, _P, _P, _I64, _I64, _I64, _I64, _P, _I32, _P, _P, _P, _SZ, _P]),
    "te_mx_gemm_fp32_scales": (ctypes.c_int, [_P, _P, _I64, _P, _P, _I64, _I32, _I64, _I64, _I64, _P, _I32, _P, _P,
                                              _P]),
    "te_mx_grouped_gemm": (ctypes.c_int, [_I32, _P, _I64, _P, _P, _I64, _P, _P, _I64, _I64, _I64, _P, _I32,
                                          _P, _P, _P, _SZ, _P]),
    "te_mx_gemm_workspace_size": (_SZ, [_I64, _I64, _I64, _I32]),
    "te_mx_device_status": (ctypes.c_int, []),
    "te_mx_selftest_timeout": (ctypes.c_int, [ctypes.c_uint32, _P]),
    "te_mx_last_error": (ctypes.c_char_p, []),
    "te_mx_version": (ctypes.c_char_p, []),
}


class TemxError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """Load libtemx.so (built in-tree by ``_build.build()``); raises if missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m mxfp8_block_scaled_quantize_gb300._build`")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(l, name)
            f.restype, f.argtypes = res, args
        _lib = l
    return _lib


def _check(status: int) -> None:
    if status != TE_MX_OK:
        raise TemxError(status, lib().te_mx_last_error().decode())


# ---------------------------------------------------------------- raw C ABI

def te_mx_scale_pitch(k: int) -> int:
    return lib().te_mx_scale_pitch(k)


def te_mx_quantize(x, rows, cols, ld_x, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col, stream) -> None:
    _check(lib().te_mx_quantize(x, rows, cols, ld_x, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col, stream))


def te_mx_block_quantize(x, rows, cols, ld_x, block_2d, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col,
                         stream) -> None:
    _check(lib().te_mx_block_quantize(x, rows, cols, ld_x, block_2d, q_row, s_row, ld_s_row, q_col, s_col,
                                      ld_s_col, stream))


def te_mx_layernorm_quantize(x, rows, hidden, ld_x, gamma, beta, eps, q_row, s_row, ld_s_row, q_col, s_col,
                             ld_s_col, mu, rsigma, stream) -> None:
    _check(lib().te_mx_layernorm_quantize(x, rows, hidden, ld_x, gamma, beta, eps, q_row, s_row, ld_s_row, q_col,
                                          s_col, ld_s_col, mu, rsigma, stream))


def te_mx_grouped_code_width(total_m, num_groups) -> int:
    return lib().te_mx_grouped_code_width(total_m, num_groups)


def te_mx_grouped_scale_width(total_m, num_groups) -> int:
    return lib().te_mx_grouped_scale_width(total_m, num_groups)


def te_mx_quantize_colwise_grouped(x, total_m, cols, ld_x, num_groups, group_m, q, ld_q, s, ld_s, stream) -> None:
    _check(lib().te_mx_quantize_colwise_grouped(x, total_m, cols, ld_x, num_groups, group_m, q, ld_q, s, ld_s,
                                                stream))


def te_mx_grouped_gemm_wgrad(num_groups, group_m, total_m, dY, s_dY, X, s_X, M, N, ld_q, ld_s, accumulate, D,
                             stream) -> None:
    _check(lib().te_mx_grouped_gemm_wgrad(num_groups, group_m, total_m, dY, s_dY, X, s_X, M, N, ld_q, ld_s,
                                          accumulate, D, stream))


def te_mx_quantize_dbias_workspace_size(rows, cols) -> int:
    return lib().te_mx_quantize_dbias_workspace_size(rows, cols)


def te_mx_quantize_dbias(x, rows, cols, ld_x, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col, dbias, workspace,
                         workspace_bytes, stream) -> None:
    _check(lib().te_mx_quantize_dbias(x, rows, cols, ld_x, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col, dbias,
                                      workspace, workspace_bytes, stream))


def te_mx_quantize_dbias_noalloc(x, rows, cols, ld_x, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col, dbias,
                                 stream) -> None:
    """Same as te_mx_quantize_dbias, for callers that cannot allocate device
    memory: the scratch is built into the library (TE_MX_NOALLOC_SCRATCH_BYTES)."""
    _check(lib().te_mx_quantize_dbias_noalloc(x, rows, cols, ld_x, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col,
                                              dbias, stream))


def te_mx_gemm(A, sA, ld_sA, B, sB, ld_sB, M, N, K, bias, epilogue, D, aux, workspace, workspace_bytes,
               stream) -> None:
    _check(lib().te_mx_gemm(A, sA, ld_sA, B, sB, ld_sB, M, N, K, bias, epilogue, D, aux, workspace,
                            workspace_bytes, stream))


def te_mx_grouped_gemm(num_groups, group_m, total_m, X, sX, ld_sX, W, sW, ld_sW, N, K, bias, epilogue, D, aux,
                       workspace, workspace_bytes, stream) -> None:
    _check(lib().te_mx_grouped_gemm(num_groups, group_m, total_m, X, sX, ld_sX, W, sW, ld_sW, N, K, bias,
                                    epilogue, D, aux, workspace, workspace_bytes, stream))


def te_mx_gemm_workspace_size(M, N, K, num_groups=0) -> int:
    return lib().te_mx_gemm_workspace_size(M, N, K, num_groups)


def te_mx_device_status() -> None:
    _check(lib().te_mx_device_status())


def te_mx_selftest_timeout(limit_us: int, stream=None) -> None:
    _check(lib().te_mx_selftest_timeout(limit_us, 0 if stream is None else stream))


def te_mx_version() -> str:
    return lib().te_mx_version().decode()


# ---------------------------------------------------------------- torch helpers

def _stream_ptr(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def quantize(x, rowwise: bool = True, colwise: bool = False, stream=None, out=None, dbias: bool = False,
             workspace=None):
    """MXFP8-quantise a 2-D bf16 CUDA tensor.  Returns a dict with q_row
    [R,C], s_row [R, pitch(C)] and/or q_col [C,R], s_col [C, pitch(R)] (uint8),
    and with ``dbias`` also "dbias" (bf16 [C], the column sums); the bias
    gradient's scratch is ``workspace`` (uint8 CUDA tensor) or allocated here."""
    import torch
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_cuda
    rows, cols = x.shape
    assert x.stride(1) == 1
    o = dict(out or {})
    if rowwise and "q_row" not in o:
        o["q_row"] = torch.empty(rows, cols, dtype=torch.uint8, device=x.device)
        o["s_row"] = torch.empty(rows, te_mx_scale_pitch(cols), dtype=torch.uint8, device=x.device)
    if colwise and "q_col" not in o:
        o["q_col"] = torch.empty(cols, rows, dtype=torch.uint8, device=x.device)
        o["s_col"] = torch.empty(cols, te_mx_scale_pitch(rows), dtype=torch.uint8, device=x.device)
    args = (x.data_ptr(), rows, cols, x.stride(0),
            _ptr(o.get("q_row")), _ptr(o.get("s_row")), o["s_row"].stride(0) if "s_row" in o else 0,
            _ptr(o.get("q_col")), _ptr(o.get("s_col")), o["s_col"].stride(0) if "s_col" in o else 0)
    if not dbias:
        te_mx_quantize(*args, _stream_ptr(stream))
        return o
    if "dbias" not in o:
        o["dbias"] = torch.empty(cols, dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = torch.empty(max(1, te_mx_quantize_dbias_workspace_size(rows, cols)), dtype=torch.uint8,
                                device=x.device)
    te_mx_quantize_dbias(*args, o["dbias"].data_ptr(), workspace.data_ptr(), workspace.numel(), _stream_ptr(stream))
    return o


def te_mx_block_scale_pitch_fp32(n) -> int:
    return int(lib().te_mx_block_scale_pitch_fp32(n))


def te_mx_block_quantize_fp32(x, rows, cols, ld_x, block_2d, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col,
                              stream) -> None:
    _check(lib().te_mx_block_quantize_fp32(x, rows, cols, ld_x, block_2d, q_row, s_row, ld_s_row, q_col, s_col,
                                           ld_s_col, stream))


def block_quantize_fp32(x, block_2d: bool = False, rowwise: bool = True, colwise: bool = False, stream=None,
                        out=None):
    """Float8BlockScaling-quantise a 2-D bf16 CUDA tensor keeping FP32 scales:
    E4M3 codes as ``block_quantize`` and fp32 scales, one per block and row
    (``s_row`` [rows, pitch(cols)], ``s_col`` [cols, pitch(rows)]), for
    ``gemm_fp32_scales``."""
    import torch
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_cuda
    rows, cols = x.shape
    assert x.stride(1) == 1
    o = dict(out or {})
    if rowwise and "q_row" not in o:
        o["q_row"] = torch.empty(rows, cols, dtype=torch.uint8, device=x.device)
        o["s_row"] = torch.empty(rows, te_mx_block_scale_pitch_fp32(cols), dtype=torch.float32, device=x.device)
    if colwise and "q_col" not in o:
        o["q_col"] = torch.empty(cols, rows, dtype=torch.uint8, device=x.device)
        o["s_col"] = torch.empty(cols, te_mx_block_scale_pitch_fp32(rows), dtype=torch.float32, device=x.device)
    te_mx_block_quantize_fp32(x.data_ptr(), rows, cols, x.stride(0), int(bool(block_2d)),
                              _ptr(o.get("q_row")), _ptr(o.get("s_row")), o["s_row"].stride(0) if "s_row" in o else 0,
                              _ptr(o.get("q_col")), _ptr(o.get("s_col")), o["s_col"].stride(0) if "s_col" in o else 0,
                              _stream_ptr(stream))
    return o


def block_quantize(x, block_2d: bool = False, rowwise: bool = True, colwise: bool = False, stream=None, out=None):
    """Float8BlockScaling-quantise a 2-D bf16 CUDA tensor with E8M0-cast
    scales: 1x128 / 128x1 blocks, or 128x128 blocks with ``block_2d``.  The
    outputs have the layout of ``quantize`` (block scales repeated per 32
    elements), so ``gemm`` consumes them as they are."""
    import torch
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_cuda
    rows, cols = x.shape
    assert x.stride(1) == 1
    o = dict(out or {})
    if rowwise and "q_row" not in o:
        o["q_row"] = torch.empty(rows, cols, dtype=torch.uint8, device=x.device)
        o["s_row"] = torch.empty(rows, te_mx_scale_pitch(cols), dtype=torch.uint8, device=x.device)
    if colwise and "q_col" not in o:
        o["q_col"] = torch.empty(cols, rows, dtype=torch.uint8, device=x.device)
        o["s_col"] = torch.empty(cols, te_mx_scale_pitch(rows), dtype=torch.uint8, device=x.device)
    te_mx_block_quantize(x.data_ptr(), rows, cols, x.stride(0), int(bool(block_2d)),
                         _ptr(o.get("q_row")), _ptr(o.get("s_row")), o["s_row"].stride(0) if "s_row" in o else 0,
                         _ptr(o.get("q_col")), _ptr(o.get("s_col")), o["s_col"].stride(0) if "s_col" in o else 0,
                         _stream_ptr(stream))
    return o


def layernorm_quantize(x, gamma, beta, eps: float = 1e-5, rowwise: bool = True, colwise: bool = False,
                       stream=None, out=None):
    """LayerNorm over the last axis of a 2-D bf16 CUDA tensor fused with its
    MXFP8 quantisation.  Returns a dict with q_row/s_row and/or q_col/s_col
    (as ``quantize``) and "mu" and "rsigma" (fp32 [rows])."""
    import torch
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_cuda and x.stride(1) == 1
    assert gamma.dtype == torch.bfloat16 and beta.dtype == torch.bfloat16
    rows, hidden = x.shape
    o = dict(out or {})
    if rowwise and "q_row" not in o:
        o["q_row"] = torch.empty(rows, hidden, dtype=torch.uint8, device=x.device)
        o["s_row"] = torch.empty(rows, te_mx_scale_pitch(hidden), dtype=torch.uint8, device=x.device)
    if colwise and "q_col" not in o:
        o["q_col"] = torch.empty(hidden, rows, dtype=torch.uint8, device=x.device)
        o["s_col"] = torch.empty(hidden, te_mx_scale_pitch(rows), dtype=torch.uint8, device=x.device)
    if "mu" not in o:
        o["mu"] = torch.empty(rows, dtype=torch.float32, device=x.device)
        o["rsigma"] = torch.empty(rows, dtype=torch.float32, device=x.device)
    te_mx_layernorm_quantize(x.data_ptr(), rows, hidden, x.stride(0), gamma.data_ptr(), beta.data_ptr(), float(eps),
                             _ptr(o.get("q_row")), _ptr(o.get("s_row")), o["s_row"].stride(0) if "s_row" in o else 0,
                             _ptr(o.get("q_col")), _ptr(o.get("s_col")), o["s_col"].stride(0) if "s_col" in o else 0,
                             _ptr(o.get("mu")), _ptr(o.get("rsigma")), _stream_ptr(stream))
    return o


def quantize_colwise_grouped(x, group_m, stream=None, out=None):
    """Per-expert column-wise MXFP8 copy of the token-major bf16 CUDA tensor x
    [total_m, cols] (experts' rows in order, ``group_m``: int32 CUDA tensor of
    token counts).  Returns {"q": uint8 [cols, ld_q], "s": uint8 [cols, ld_s]}
    in the padded per-expert layout (widths from te_mx_grouped_*_width)."""
    import torch
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_cuda and x.stride(1) == 1
    assert group_m.dtype == torch.int32 and group_m.is_cuda
    total_m, cols = x.shape
    G = group_m.numel()
    o = dict(out or {})
    if "q" not in o:
        o["q"] = torch.empty(cols, te_mx_grouped_code_width(total_m, G), dtype=torch.uint8, device=x.device)
        o["s"] = torch.empty(cols, te_mx_grouped_scale_width(total_m, G), dtype=torch.uint8, device=x.device)
    te_mx_quantize_colwise_grouped(x.data_ptr(), total_m, cols, x.stride(0), G, group_m.data_ptr(), o["q"].data_ptr(),
                                   o["q"].stride(0), o["s"].data_ptr(), o["s"].stride(0), _stream_ptr(stream))
    return o


def grouped_gemm_wgrad(group_m, total_m, dy, x, stream=None, out=None, accumulate: bool = False):
    """dW_e = dY_e^T X_e for every expert: ``dy`` and ``x`` are the dicts of
    quantize_colwise_grouped of dY [total_m, M] and X [total_m, N] (same
    group_m).  Returns bf16 [G, M, N] (``out`` if given); with ``accumulate``,
    ``out`` is an fp32 [G, M, N] tensor that is added to."""
    import torch
    G = group_m.numel()
    M, N = dy["q"].shape[0], x["q"].shape[0]
    assert dy["q"].stride(0) == x["q"].stride(0) and dy["s"].stride(0) == x["s"].stride(0)
    if accumulate:
        assert out is not None and out.dtype == torch.float32
    d = out if out is not None else torch.empty(G, M, N, dtype=torch.bfloat16, device=dy["q"].device)
    te_mx_grouped_gemm_wgrad(G, group_m.data_ptr(), total_m, dy["q"].data_ptr(), dy["s"].data_ptr(), x["q"].data_ptr(),
                             x["s"].data_ptr(), M, N, dy["q"].stride(0), dy["s"].stride(0), int(bool(accumulate)),
                             d.data_ptr(), _stream_ptr(stream))
    return d


def gemm(qa, sa, qb, sb, bias=None, gelu: bool = False, stream=None, out=None, dgelu_aux=None,
         accumulate=None):
    """D = epilogue(deq(qa) . deq(qb)^T (+ bias)) in bf16; returns (D, aux or None).
    With ``dgelu_aux`` (bf16 [M, N], the forward pre-activation) the epilogue is
    D = bf16(acc * gelu'(dgelu_aux)).  With ``accumulate`` (an fp32 [M, N] CUDA
    tensor) it is accumulate += deq(qa) . deq(qb)^T in fp32."""
    import torch
    M, K = qa.shape
    N = qb.shape[0]
    if accumulate is not None:
        assert accumulate.dtype == torch.float32 and bias is None and not gelu and dgelu_aux is None
        te_mx_gemm(qa.data_ptr(), sa.data_ptr(), sa.stride(0), qb.data_ptr(), sb.data_ptr(), sb.stride(0),
                   M, N, K, 0, EPI_ACCUMULATE_F32, accumulate.data_ptr(), 0, 0, 0, _stream_ptr(stream))
        return accumulate, None
    epi = (EPI_BIAS if bias is not None else EPI_NONE) + (EPI_GELU_AUX if gelu else 0)
    if dgelu_aux is not None:
        assert bias is None and not gelu
        d = torch.empty(M, N, dtype=torch.bfloat16, device=qa.device) if out is None else out[0]
        te_mx_gemm(qa.data_ptr(), sa.data_ptr(), sa.stride(0), qb.data_ptr(), sb.data_ptr(), sb.stride(0),
                   M, N, K, 0, EPI_DGELU, d.data_ptr(), dgelu_aux.data_ptr(), 0, 0, _stream_ptr(stream))
        return d, None
    if out is None:
        d = torch.empty(M, N, dtype=torch.bfloat16, device=qa.device)
        aux = torch.empty(M, N, dtype=torch.bfloat16, device=qa.device) if gelu else None
    else:
        d, aux = out
    te_mx_gemm(qa.data_ptr(), sa.data_ptr(), sa.stride(0), qb.data_ptr(), sb.data_ptr(), sb.stride(0),
               M, N, K, _ptr(bias), epi, d.data_ptr(), _ptr(aux), 0, 0, _stream_ptr(stream))
    return d, aux


def te_mx_gemm_fp32_scales(A, sA, ld_sA, B, sB, ld_sB, b_blocks_2d, M, N, K, bias, epilogue, D, aux,
                           stream) -> None:
    _check(lib().te_mx_gemm_fp32_scales(A, sA, ld_sA, B, sB, ld_sB, b_blocks_2d, M, N, K, bias, epilogue, D, aux,
                                        stream))


def gemm_fp32_scales(qa, sa, qb, sb, b_blocks_2d: bool, bias=None, gelu: bool = False, stream=None, out=None,
                     dgelu_aux=None):
    """Float8BlockScaling GEMM with FP32 scales (``block_quantize_fp32``
    output; ``b_blocks_2d`` for 128x128 weight blocks): D = epilogue(sum over
    128-long K blocks of sA sB A_kb . B_kb^T (+ bias)); returns (D, aux or None).
    With ``dgelu_aux`` the epilogue is the GELU backward (see ``gemm``)."""
    import torch
    M, K = qa.shape
    N = qb.shape[0]
    epi = (EPI_BIAS if bias is not None else EPI_NONE) + (EPI_GELU_AUX if gelu else 0)
    aux = None
    if dgelu_aux is not None:
        assert bias is None and not gelu
        epi = EPI_DGELU
    if out is None:
        d = torch.empty(M, N, dtype=torch.bfloat16, device=qa.device)
        if gelu:
            aux = torch.empty(M, N, dtype=torch.bfloat16, device=qa.device)
    else:
        d, aux = out
    aux_ptr = dgelu_aux.data_ptr() if dgelu_aux is not None else _ptr(aux)
    te_mx_gemm_fp32_scales(qa.data_ptr(), sa.data_ptr(), sa.stride(0), qb.data_ptr(), sb.data_ptr(), sb.stride(0),
                           int(bool(b_blocks_2d)), M, N, K, _ptr(bias), epi, d.data_ptr(), aux_ptr,
                           _stream_ptr(stream))
    return d, (aux if dgelu_aux is None else None)


def grouped_gemm(group_m, qx, sx, qw, sw, bias=None, gelu: bool = False, stream=None, out=None, dgelu_aux=None):
    """Grouped GEMM over experts: group_m int32 [G] on the device, qx [total_m, K],
    qw [G, N, K], sw [G*N, pitch]; returns (D, aux or None) of [total_m, N].
    With ``dgelu_aux`` the epilogue is the GELU backward (see ``gemm``)."""
    import torch
    total_m, K = qx.shape
    G, N, _ = qw.shape
    epi = (EPI_BIAS if bias is not None else EPI_NONE) + (EPI_GELU_AUX if gelu else 0)
    if dgelu_aux is not None:
        assert bias is None and not gelu
        d = torch.empty(total_m, N, dtype=torch.bfloat16, device=qx.device) if out is None else out[0]
        sw2 = sw.reshape(G * N, -1)
        te_mx_grouped_gemm(G, group_m.data_ptr(), total_m, qx.data_ptr(), sx.data_ptr(), sx.stride(0),
                           qw.data_ptr(), sw2.data_ptr(), sw2.stride(0), N, K, 0, EPI_DGELU,
                           d.data_ptr(), dgelu_aux.data_ptr(), 0, 0, _stream_ptr(stream))
        return d, None
    if out is None:
        d = torch.empty(total_m, N, dtype=torch.bfloat16, device=qx.device)
        aux = torch.empty(total_m, N, dtype=torch.bfloat16, device=qx.device) if gelu else None
    else:
        d, aux = out
    sw2 = sw.reshape(G * N, -1)
    te_mx_grouped_gemm(G, group_m.data_ptr(), total_m, qx.data_ptr(), sx.data_ptr(), sx.stride(0),
                       qw.data_ptr(), sw2.data_ptr(), sw2.stride(0), N, K, _ptr(bias), epi,
                       d.data_ptr(), _ptr(aux), 0, 0, _stream_ptr(stream))
    return d, aux
