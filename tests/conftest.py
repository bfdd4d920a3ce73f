import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    # A fresh checkout has neither library (both build folders are ignored by
    # git): build them once here when nvcc is available, so the test modules
    # can load them.  Nothing is built when they already exist.
    import shutil
    lib = os.path.join(ROOT, "block_scaled_fp8_group_gb300", "_build", "libfp8bq.so")
    if not os.path.exists(lib) and shutil.which("nvcc"):
        from block_scaled_fp8_group_gb300 import build as package_build
        package_build.build()
    orc = os.path.join(ROOT, "oracle", "_build", "liboracle.so")
    if not os.path.exists(orc) and shutil.which("gcc"):
        import oracle
        oracle.build()
