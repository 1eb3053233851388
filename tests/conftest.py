import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture
def pin_kernels():
    """pin_kernels(attention="one_tile" | "two_tile", one_tile_keys=, gemm_bn=, lib=)
    pins the library's kernel choices for one test (sdpa_set_kernel_choice)
    and returns them to the shapes when the test ends."""
    import transformer_scaled_dot_02_gb300 as sd
    pinned = []

    def pin(attention=None, one_tile_keys=0, gemm_bn=0, lib=None):
        sd.sdpa_set_kernel_choice(sd.ATTENTION_KERNELS[attention], one_tile_keys, gemm_bn, lib=lib)
        pinned.append(lib)

    yield pin
    for lib in pinned:
        sd.sdpa_set_kernel_choice(0, 0, 0, lib=lib)
