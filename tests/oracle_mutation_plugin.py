"""pytest plugin for tests/test_oracle_mutations.py: replaces one oracle function (named by
QW_ORACLE_MUTATE="module:function") with a copy whose result has one element changed, so
that the oracle's CPU pins can be shown to catch it.  Test infrastructure only."""
import functools
import importlib
import os
import sys

import numpy as np


def perturb(x):
    """The same result with its first element changed (by far more than any tolerance)."""
    if isinstance(x, tuple):
        return (perturb(x[0]),) + x[1:]
    if isinstance(x, list):
        return [perturb(x[0])] + x[1:] if x else x
    if isinstance(x, np.ndarray):
        y = np.array(x, copy=True)
        if y.size == 0:
            return y
        flat = y.reshape(-1)
        if y.dtype == np.bool_:
            flat[0] = ~flat[0]
        elif np.issubdtype(y.dtype, np.integer):
            flat[0] = flat[0] + 1
        else:
            flat[0] = flat[0] + 1.0 + 2 * np.max(np.abs(np.nan_to_num(flat)))
        return y
    if isinstance(x, (bool, np.bool_)):
        return not x
    if isinstance(x, (int, np.integer)):
        return x + 1
    if isinstance(x, (float, np.floating)):
        return x + 1.0 + abs(x)
    return x


def pytest_configure(config):
    spec = os.environ.get("QW_ORACLE_MUTATE")
    if not spec:
        return
    modname, name = spec.split(":")
    mod = importlib.import_module(modname)
    orig = getattr(mod, name)

    @functools.wraps(orig)
    def mutated(*a, **k):
        return perturb(orig(*a, **k))

    setattr(mod, name, mutated)
    # modules that imported the function by name
    for m in list(sys.modules.values()):
        if m is not None and getattr(m, name, None) is orig:
            setattr(m, name, mutated)
