import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built extension")


def pytest_sessionstart(session):
    """RLHEAD_GEMM_PAIR=0/1 selects the single-SM or SM-pair tensor-core GEMMs for a run."""
    v = os.environ.get("RLHEAD_GEMM_PAIR")
    if v is None:
        return
    try:
        import lm_head_gb300 as rh
        from lm_head_gb300 import build
        build.build()
        rh.rl_set_option(rh.RL_OPT_GEMM_PAIR, int(v))
    except Exception:
        pass
