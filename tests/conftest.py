import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    # Build the CUDA library and the C oracle if they are missing or stale,
    # so that importing the package (which loads liblinattn.so) works.
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_la_build", os.path.join(ROOT, "linear_attention_02_gb300", "build.py"))
    nb = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(nb)
    nb.build()
    import oracle
    oracle.build()
