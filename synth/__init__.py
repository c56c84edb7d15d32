"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This package draws random numbers and lays them out in the canonical input
formats of the library (packed integer words, E2M1 nibbles, E8M0 bytes, BF16
and E4M3 bit patterns).  It contains no dequantization, no GEMM and no routing
arithmetic: those live, independently, in ``oracle/`` (CPU reference) and in
the CUDA library (``moe_qw_repack_gb300``).
"""
from .gen import *  # noqa: F401,F403
