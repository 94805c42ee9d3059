"""Rotation-based W4A4 inference kernels for GB300 (sm_103a).

The compute lives in ``librq.so`` (CUDA kernels behind the C ABI declared in
``include/rq.h``).  This package only marshals arguments: tensors in, device
pointers, sizes and the current CUDA stream out.  There is no fallback: if the
library cannot be loaded, every call raises.

Entry points (same names as the C ABI):

* :func:`fwht_quant` -- randomized Hadamard rotation of each row + per-row INT4
  quantization and nibble packing (also the offline weight fold when given W^T);
* :func:`w4a4_gemm` -- exact INT4 x INT4 product with per-token x per-channel
  dequant (or per-group weight scales on the operand-form activations that
  :func:`fwht_quant` writes with ``RQ_E4M3_CODES``);
* :func:`kv_rotate_quant` -- head-wise rotation + INT4 quantization of K and V;
* :func:`fwht_quant_gemm` -- decode-sized fusion of the rotation, quantization
  and W4A4 product in one launch;
* :func:`attn_decode` -- attention of decode queries over the rotated INT4 KV
  cache;
* :func:`w4a8_gemm` -- the W4A8 linear layer (INT8 activations from
  :func:`fwht_quant` with ``RQ_INT8_CODES``), per-channel or per-group weight
  scales;
* :func:`sync_status` -- drain a stream and read (and clear) the device error
  word that bounded waits raise; :func:`selftest_wait_timeout` makes one such
  wait run out on purpose, to exercise that path;
* :func:`probe_f8_mma` -- a measurement aid: back-to-back FP8 MMAs on every SM,
  the rate of the tensor pipe the W4A4 products run on.
"""
from ._binding import (  # noqa: F401
    RQ_A_E4M3,
    RQ_ATTN_ROTATED_OUT,
    RQ_E4M3_CODES,
    RQ_GROUP_SCALES,
    RQ_INT4_BYTES,
    RQ_INT8_CODES,
    RQ_SIGNS_FIRST,
    RQError,
    attn_decode,
    fwht_quant,
    fwht_quant_gemm,
    kv_rotate_quant,
    library_path,
    load_library,
    probe_f8_mma,
    selftest_wait_timeout,
    sync_status,
    w4a4_gemm,
    w4a8_gemm,
)

__all__ = ["RQ_A_E4M3", "RQ_ATTN_ROTATED_OUT", "RQ_E4M3_CODES", "RQ_GROUP_SCALES", "RQ_INT4_BYTES", "RQ_INT8_CODES", "RQ_SIGNS_FIRST", "RQError", "attn_decode",
           "fwht_quant", "fwht_quant_gemm", "kv_rotate_quant", "library_path", "load_library", "probe_f8_mma", "selftest_wait_timeout",
           "sync_status",
           "w4a4_gemm", "w4a8_gemm"]
