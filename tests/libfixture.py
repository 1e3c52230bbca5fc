"""Builds (if stale) and loads libpagedkv.so for the tests."""
import pytest


@pytest.fixture(scope="session")
def palib():
    from paged_kv_cache_191_gb300 import build, ops
    build.build()
    return ops.lib()
