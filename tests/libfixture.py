"""Builds libchunk_attention.so once per test session (host C++ and sm_103a
kernels; cross-compiles without a GPU)."""
import pytest


@pytest.fixture(scope="session")
def lib():
    from prefix_shared_decode_gb300 import build, capi
    build.build()
    return capi.lib()
