"""CPU oracle for the quantized-GEMM hot path (test infrastructure only).

Plain, slow, float64 restatements of what the library computes, written from the
Humming pages ("quantized推論のための高速かつ柔軟なカーネル「Humming」を発表",
spke.com; and "vLLM Humming performance benchmark", aireiter.com) and the public
format definitions they name.  It shares no code, table or constant with the CUDA
library and never imports it.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline and
``--impl reference`` legs) may import this package.  The product path must not.

Pin status of every function (what checks it against something other than itself)
is listed in each module's docstring; nothing here is "parity unpinned".
"""
from . import act, formats, qgemm, moe  # noqa: F401
