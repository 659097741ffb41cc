"""The C-ABI library builds, loads and exports every entry point declared in
include/dspark.h; host-side validation rejects bad arguments before any CUDA call
(runs without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from draft_sampling_verification_tcgen05_gb300 import _build
    _build.build()
    import draft_sampling_verification_tcgen05_gb300 as ds
    return ds.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "dspark.h")).read()
    return re.findall(r"DSPARK_API\s+[\w\s\*]+?\b(dspark_\w+)\s*\(", text)


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    for op in ("dspark_draft_logits", "dspark_markov_sample", "dspark_verify", "dspark_schedule",
               "dspark_verify_greedy", "dspark_confidence", "dspark_markov_sample_reduced",
               "dspark_verify_logits", "dspark_verify_gumbel", "dspark_markov_sample_conf"):
        assert op in names


def test_workspace_sizes(L):
    assert L.dspark_workspace_size(0, 0, 0, 0, 0) == 256
    # header, per-request segment counters, per-segment masses
    assert L.dspark_workspace_size(2, 256, 8, 151936, 0) == 256 + 1024 + 8 * 256 * 297
    m = L.dspark_workspace_size(1, 64, 16, 151936, 256)
    assert m >= 256 + 64 * 16 * 12
    assert L.dspark_workspace_size(3, 1024, 16, 0, 0) == 256 + 2 * 8 * 1024 * 16
    assert L.dspark_workspace_size(4, 256, 8, 151936, 0) == 256 + 8 * 256 * 9 + 1024
    assert L.dspark_workspace_size(5, 64, 16, 151936, 256) == 256
    vl = L.dspark_workspace_size(6, 256, 8, 151936, 256)
    # keys, per-request and per-row counters, window masks, per-round counts, decisions, row
    # selections, two request lists, the window's normalisers and chunk partials (one row per
    # round at this size)
    assert vl == 256 + 2048 + 1024 + 1024 + 8192 + 1024 + 1024 + 256 + 1024 + 8192 + 2048 + 1024 + 8 * 256 * 75
    assert L.dspark_workspace_size(6, 0, 8, 100, 8) == 0
    assert L.dspark_workspace_size(7, 256, 8, 151936, 0) == 256 + 8 * 256 * 9 + 1024
    assert L.dspark_workspace_size(9, 1, 1, 1, 1) == 0


def test_host_validation_without_gpu(L):
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(4096)        # never dereferenced: validation fails first
    assert L.dspark_draft_logits(null, fake, 1, 8, 64, 100, fake, fake, 256, null) == 1
    assert L.dspark_draft_logits(fake, fake, 1, 8, 60, 100, fake, fake, 256, null) == 1   # H*2 % 16
    assert L.dspark_draft_logits(fake, fake, 7, 8, 64, 100, fake, fake, 256, null) == 1   # dtype
    assert L.dspark_draft_logits(fake, fake, 1, 8, 64, 100, fake, fake, 16, null) == 1    # workspace
    assert L.dspark_markov_sample(fake, fake, fake, fake, 1, fake, 0, 2 ** 32, 1, 8, 100, 64,
                                  fake, null, fake, 1 << 20, null) == 1                   # offset
    assert L.dspark_markov_sample(fake, fake, fake, fake, 1, fake, 0, 0, 1, 0, 100, 64,
                                  fake, null, fake, 1 << 20, null) == 1                   # N = 0
    assert L.dspark_verify(fake, fake, fake, null, 0, 0, 1, 0, 10, fake, fake, fake, 256, null) == 1
    # the sampler with the confidence head: a missing head pointer or an unknown hidden dtype is refused
    L.dspark_markov_sample_conf.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.c_void_p, ctypes.c_uint64,
                                            ctypes.c_uint64] + [ctypes.c_int] * 4 + [ctypes.c_void_p, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float] + \
        [ctypes.c_void_p] * 5 + [ctypes.c_size_t, ctypes.c_void_p]
    assert L.dspark_markov_sample_conf(fake, fake, fake, fake, 1, fake, 0, 0, 1, 8, 100, 64, fake, 1, 256, fake, null,
                                       0.5, fake, fake, fake, null, fake, 1 << 20, null) == 1
    assert L.dspark_markov_sample_conf(fake, fake, fake, fake, 1, fake, 0, 0, 1, 8, 100, 64, fake, 7, 256, fake, fake,
                                       0.5, fake, fake, fake, null, fake, 1 << 20, null) == 1
    assert L.dspark_markov_sample_reduced(fake, fake, fake, fake, 1, fake, 0, 0, 1, 8, 100, 64, null, 0, 500,
                                          fake, null, fake, 1 << 20, null) == 1                # no table
    assert L.dspark_markov_sample_reduced(fake, fake, fake, fake, 1, fake, 0, 0, 1, 8, 100, 64, fake, 2, 500,
                                          fake, null, fake, 1 << 20, null) == 1                # mode
    assert L.dspark_verify_greedy(fake, fake, null, 1, 0, 10, fake, fake, fake, 1 << 20, null) == 1  # gamma = 0
    assert L.dspark_verify_greedy(null, fake, null, 1, 2, 10, fake, fake, fake, 1 << 20, null) == 1
    assert L.dspark_verify_greedy(fake, fake, null, 4, 8, 10, fake, fake, fake, 64, null) == 1      # workspace
    vl = [fake, fake, fake, fake, fake, fake, 1, 64, fake, fake, fake, null, 0, 0, 4, 8, 1000, fake, fake, fake,
          1 << 30, null]

    def vl_with(**kw):
        args = list(vl)
        for i, v in kw.items():
            args[int(i[1:])] = v
        return L.dspark_verify_logits(*args)

    assert vl_with(a6=2) == 1                                                # dtype
    assert vl_with(a7=4) == 1                                                # r * 2 bytes not a multiple of 16
    assert vl_with(a7=2048) == 1                                             # r too large
    assert vl_with(a13=2 ** 32) == 1                                         # offset
    assert vl_with(a15=0) == 1                                               # gamma = 0
    assert vl_with(a9=null) == 1                                             # no draft lse
    assert vl_with(a0=ctypes.c_void_p(4100)) == 1                            # misaligned logits
    assert vl_with(a20=1024) == 1                                            # workspace
    vg = [fake, fake, fake, null, 0, 0, 4, 8, 1000, fake, fake, fake, 1 << 20, null]

    def vg_with(**kw):
        args = list(vg)
        for i, v in kw.items():
            args[int(i[1:])] = v
        return L.dspark_verify_gumbel(*args)

    assert vg_with(a1=null) == 1                                             # no temperature
    assert vg_with(a5=2 ** 32) == 1                                          # offset
    assert vg_with(a7=0) == 1                                                # gamma = 0
    assert vg_with(a8=1 << 27) == 1                                          # V too large
    assert vg_with(a0=ctypes.c_void_p(4100)) == 1                            # misaligned logits
    assert vg_with(a12=64) == 1                                              # workspace
    assert L.dspark_confidence(fake, 1, fake, 1, fake, fake, fake, fake, 0.0, fake, 1, 8, 64, 100, 0,
                               fake, fake, 256, null) == 1                                   # r = 0
    assert L.dspark_confidence(fake, 3, fake, 1, fake, fake, fake, fake, 0.0, fake, 1, 8, 64, 100, 8,
                               fake, fake, 256, null) == 1                                   # dtype
    assert L.dspark_schedule(fake, null, 0, 4, 4, -1, fake, fake, fake, fake, fake, 1024, null) == 1
    assert L.dspark_schedule(fake, null, 0, 2048, 1024, 5, fake, fake, fake, fake, fake, 1 << 30, null) == 1
    assert b"SPS" in L.dspark_last_error() or len(L.dspark_last_error()) > 0
    assert L.dspark_status_string(4) == b"device wait timed out"


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import draft_sampling_verification_tcgen05_gb300 as ds
    monkeypatch.setattr(ds, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(ds, "_lib", None)
    with pytest.raises(RuntimeError):
        ds.lib()
