"""The product path has no fallback: without the built library every call
raises, and nothing in the package reaches the oracle.  Host only."""
import ast
import os

import pytest

from paged_kv_cache_191_gb300 import ops

PKG = os.path.dirname(ops.__file__)


@pytest.fixture
def no_library(monkeypatch, tmp_path):
    monkeypatch.setattr(ops, "LIB_PATH", str(tmp_path / "libpagedkv.so"))
    monkeypatch.setattr(ops, "_lib", None)


def test_missing_library_raises(no_library):
    with pytest.raises(RuntimeError, match="missing"):
        ops.lib()


def test_host_block_manager_needs_the_library(no_library):
    with pytest.raises(RuntimeError, match="missing"):
        ops.BlockAllocator(8)


def test_scheduler_needs_the_library(no_library):
    with pytest.raises(RuntimeError, match="missing"):
        ops.Scheduler(num_blocks=8, max_batch=2, max_tokens=32, host_blocks=0)


def _imports(path):
    tree = ast.parse(open(path).read(), path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            yield from (a.name for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            yield node.module or ""


def test_package_never_imports_the_oracle():
    sources = [os.path.join(PKG, f) for f in os.listdir(PKG) if f.endswith(".py")]
    assert sources
    for path in sources:
        mods = list(_imports(path))
        assert not any(m == "oracle" or m.startswith("oracle.") for m in mods), path
