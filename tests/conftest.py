import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def _ensure_library():
    # The binding fails loudly without the compiled library; build it in-tree
    # once if this checkout has not been built yet.
    lib = os.path.join(ROOT, "linear_attention_state_chunked_gb300", "liblinstate.so")
    if not os.path.exists(lib):
        import __graft_entry__
        __graft_entry__.build()


_ensure_library()
