import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libgdn")


def _ensure_built():
    """The ABI tests load libgdn.so; build it in-tree when it is absent or stale."""
    here = os.path.join(ROOT, "gated_delta_rule_backward_gb300")
    lib = os.path.join(here, "libgdn.so")
    srcs = [os.path.join(here, "csrc", f) for f in os.listdir(os.path.join(here, "csrc"))]
    srcs.append(os.path.join(ROOT, "include", "gdn.h"))
    if not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(s) for s in srcs):
        from gated_delta_rule_backward_gb300 import build
        build.build()


_ensure_built()
