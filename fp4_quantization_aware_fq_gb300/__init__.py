"""GB300-native block-scaled FP4 fake-quantization (NVFP4, MXFP4, double-block
NVFP4; nearest-even and stochastic rounding; STE mask; OsciReset statistics;
random Hadamard transform of backward operands; static outlier retention;
the QAD distillation loss; the block-scaled FP4 GEMM on the tensor cores).

The compute lives in the CUDA library built from ``csrc/`` (C ABI in
``include/fq.h``); ``fq`` is its Python binding.  Importing this package does
not load the library; the first call does, and fails loudly if it is absent.
"""
from .fq import (BF16, COL, F32, MXFP4, NVFP4, NVFP4_2LEVEL, RNE, ROW, ROWCOL, SR, Config,
                 FqError, Outliers, QTensor, alloc_qtensor, fq_amax, fq_channel_amax,
                 fq_dequantize, fq_gemm, fq_gemm_workspace_size, fq_fakequant_ste, fq_osci_reset, fq_osci_update,
                 fq_osci_update_noalloc, fq_osci_update_reset, fq_osci_workspace_size,
                 fq_qad_kl, fq_quantize, fq_quantize_outliers, fq_select_channels, fq_status_string,
                 fq_ste_backward, fq_workspace_size)

__all__ = ["BF16", "COL", "F32", "MXFP4", "NVFP4", "NVFP4_2LEVEL", "RNE", "ROW", "ROWCOL", "SR",
           "Config", "FqError", "Outliers", "QTensor", "alloc_qtensor", "fq_amax",
           "fq_channel_amax", "fq_dequantize", "fq_gemm", "fq_gemm_workspace_size", "fq_fakequant_ste", "fq_osci_reset",
           "fq_osci_update", "fq_osci_update_noalloc", "fq_osci_update_reset",
           "fq_osci_workspace_size", "fq_qad_kl", "fq_quantize", "fq_quantize_outliers",
           "fq_select_channels", "fq_status_string", "fq_ste_backward", "fq_workspace_size"]
