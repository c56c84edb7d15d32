"""GB300-native low-bit weight-quantized GEMM (W4A16 INT4/INT3, W4A8 MXFP4 x MXFP8) for
dense and MoE layers, behind the C ABI of include/qw.h.

``moe_qw_repack_gb300.qw`` is the Python binding (loads ``_build/libqw.so``);
``moe_qw_repack_gb300.build`` compiles it for sm_103a.
"""
__all__ = ["qw", "build"]
