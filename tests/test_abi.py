"""CPU-side checks of the C ABI: the library builds, loads and exports every symbol that
include/dspark.h declares, the binding declares each of them, and host-side validation rejects
bad arguments before touching the GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from semi_autoregressive_drafting_gb300 import _build, _lib
    _build.build()
    return _lib.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "dspark.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ["dspark_markov_draft", "dspark_rnn_draft", "dspark_confidence",
              "dspark_tv_label", "dspark_prefix_schedule", "dspark_workspace_bytes",
              "dspark_get_status", "dspark_last_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from semi_autoregressive_drafting_gb300 import _lib
    for name in _declared():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding does not declare {name}"


def test_no_torch_in_the_abi():
    src = open(os.path.join(ROOT, "include", "dspark.h")).read()
    assert "torch" not in src.lower().replace("pytorch", "")
    assert "#include <cuda" not in src          # plain C header: no CUDA types either


def test_host_validation_without_gpu(lib):
    V, r = 4096, 64
    p = ctypes.c_void_p(16)
    args = lambda B, G, V, r, d, T, lay=0: (B, G, V, r, d, T, 0, 0, p, p, lay, None, 0, p, None, p,
                                            None, None, p, p, None, None, None, None, None, p,
                                            1 << 20, None)
    assert lib.dspark_markov_draft(*args(0, 7, V, r, 0, 1.0)) == 1      # B = 0
    assert lib.dspark_markov_draft(*args(1, 17, V, r, 0, 1.0)) == 1     # gamma > 16
    assert lib.dspark_markov_draft(*args(1, 7, V, 60, 0, 1.0)) == 1     # r not a multiple of 8
    assert lib.dspark_markov_draft(*args(1, 7, V, r, 0, 0.0)) == 1      # T = 0
    assert lib.dspark_markov_draft(*args(1, 7, V, r, 0, float("nan"))) == 1
    assert b"T must be" in lib.dspark_last_error()
    assert lib.dspark_markov_draft(*args(1, 7, V, r, 0, 1.0, 2)) == 1   # unknown W2 layout
    assert b"W2 layout" in lib.dspark_last_error()
    assert lib.dspark_prefix_schedule(1000, 17, p, p, p, p, None) == 1
    assert lib.dspark_tv_label(0, 10, 1.0, p, p, p, None, None) == 1


def test_path_override(lib, monkeypatch):
    monkeypatch.setenv("DSPARK_DRAFT_PATH", "cuda-core")
    assert lib.dspark_draft_path(0, 1, 151936, 256, 1) == 0
    monkeypatch.setenv("DSPARK_DRAFT_PATH", "tensor")
    assert lib.dspark_draft_path(0, 1, 151936, 256, 1) == 1
    monkeypatch.setenv("DSPARK_DRAFT_PATH", "tensor-vocab")
    assert lib.dspark_draft_path(0, 4, 151936, 72, 1) == -1      # that kernel cannot run it
    assert lib.dspark_draft_path(0, 8, 151936, 256, 1) == -1
    monkeypatch.setenv("DSPARK_DRAFT_PATH", "something-else")     # unknown: automatic choice
    assert lib.dspark_draft_path(0, 1, 151936, 256, 1) == 0
    assert lib.dspark_draft_path(0, 4, 151936, 256, 1) == 2


def test_cluster_query_without_device(lib):
    # the query needs a device for the SM layout: negative here, and for rejected arguments
    assert lib.dspark_draft_cluster(0, 1, 151936, 250, 1) < 0


def test_path_selection(lib, monkeypatch):
    monkeypatch.delenv("DSPARK_DRAFT_PATH", raising=False)
    from semi_autoregressive_drafting_gb300 import _lib
    assert lib.dspark_draft_path(0, 1, 151936, 256, 1) == 0      # latency regime: CUDA cores
    assert lib.dspark_draft_path(0, 2, 151936, 256, 1) == 0
    assert lib.dspark_draft_path(0, 3, 151936, 256, 1) == 2      # tensor cores, vocabulary on M
    assert lib.dspark_draft_path(0, 4, 151936, 72, 1) == 0       # rank not in 64-blocks: CUDA cores
    assert lib.dspark_draft_path(0, 4, 4096, 64, 0) == 0
    assert lib.dspark_draft_path(0, 1, 151936, 250, 1) == -1     # invalid rank


def test_launch_counts(lib, monkeypatch):
    monkeypatch.delenv("DSPARK_DRAFT_PATH", raising=False)
    assert lib.dspark_draft_launches(0, 1, 151936, 256, 1) == 1     # one persistent launch
    assert lib.dspark_draft_launches(1, 128, 151936, 256, 1) == 2   # + the RNN head's h-part GEMM
    assert lib.dspark_draft_launches(0, 1, 151936, 250, 1) == -1
    assert lib.dspark_draft_loss_launches(64, 7, 151936, 1) == 4    # three phases + totals
    assert lib.dspark_draft_loss_launches(64, 7, 151936, 0) == 3    # no gradient pass
    assert lib.dspark_draft_loss_launches(0, 7, 151936, 1) == -1
    assert lib.dspark_draft_loss_launches(1, 17, 151936, 1) == -1
    assert lib.dspark_draft_loss_launches(1, 7, 1, 1) == -1
