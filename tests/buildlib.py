"""Build the CUDA library and the oracle in place before tests import them.
The build script is loaded by file path: importing the package itself
requires the built library."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_done = False


def ensure_built():
    global _done
    if _done:
        return
    spec = importlib.util.spec_from_file_location(
        "ssm_build", os.path.join(ROOT, "selective_state_space_123_b300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    import oracle
    oracle.build()
    _done = True
