"""Every public oracle function is pinned: with one element of its result changed, some
CPU test of the oracle fails.  Each function is mutated in a fresh pytest process
(tests/oracle_mutation_plugin.py) that runs the oracle's own CPU tests."""
import importlib
import inspect
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MODULES = ["oracle.formats", "oracle.qgemm", "oracle.moe", "oracle.act"]
PIN_FILES = ["tests/test_oracle_formats.py", "tests/test_oracle_gemm.py",
             "tests/test_oracle_moe.py", "tests/test_oracle_route.py",
             "tests/test_oracle_act.py", "tests/test_oracle_fp4_int1.py"]


def oracle_functions():
    out = []
    for m in MODULES:
        mod = importlib.import_module(m)
        for name, f in inspect.getmembers(mod, inspect.isfunction):
            if f.__module__ == m and not name.startswith("_"):
                out.append(f"{m}:{name}")
    return out


def test_every_oracle_function_is_listed():
    assert len(oracle_functions()) >= 40


def run_mutated(spec):
    env = dict(os.environ, QW_ORACLE_MUTATE=spec,
               PYTHONPATH=os.pathsep.join([os.path.join(ROOT, "tests"), ROOT]))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu",
                        "-p", "oracle_mutation_plugin", "-p", "no:cacheprovider", *PIN_FILES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    return spec, r.returncode, r.stdout[-300:]


def test_a_planted_mutation_fails_a_pin():
    """One fresh pytest process per function, several at a time; exit status 1 = a pin
    failed (the mutation was caught)."""
    import concurrent.futures as cf
    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(run_mutated, oracle_functions()))
    missed = [(spec, rc, out) for spec, rc, out in results if rc != 1]
    assert not missed, "mutations that no pin caught: " + repr(missed)
