import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libq4.so")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes of CPU oracle time)")


def _lib_stale() -> bool:
    pkg = os.path.join(ROOT, "int4_weight_only_q4_gb300")
    so = os.path.join(pkg, "libq4.so")
    if not os.path.exists(so):
        return True
    srcs = [os.path.join(pkg, "csrc", f) for f in os.listdir(os.path.join(pkg, "csrc"))]
    srcs.append(os.path.join(ROOT, "include", "q4.h"))
    return any(os.path.getmtime(s) > os.path.getmtime(so) for s in srcs)


def pytest_sessionstart(session):
    # the library under test is built in-tree from the committed sources
    if _lib_stale():
        import importlib.util
        spec = importlib.util.spec_from_file_location(
            "_q4_build", os.path.join(ROOT, "int4_weight_only_q4_gb300", "build.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod.build()
