"""The C-ABI library loads and exports every entry point declared in include/dspark.h.

Runs without a GPU: nothing here launches work.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "dspark.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_draft_gb300 import build
    build.build()
    import speculative_decoding_draft_gb300 as ds
    return ds.lib()


def test_header_declares_the_three_operations():
    names = _declared()
    for op in ("dspark_draft_markov_sample", "dspark_schedule_survival", "dspark_verify_ragged"):
        assert op in names


def test_every_declared_symbol_is_exported(lib):
    import speculative_decoding_draft_gb300 as ds
    names = _declared()
    assert set(names) == set(ds.EXPORTED_SYMBOLS)
    for name in names:
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    import speculative_decoding_draft_gb300 as ds
    assert lib.dspark_version() == 200
    for code, name in ds.STATUS_NAMES.items():
        assert ds.status_string(code) == name


def test_workspace_queries(lib):
    import speculative_decoding_draft_gb300 as ds
    base = ds.draft_workspace_bytes(2048, 7, 151936, 256, ds.BF16, ds.FLAG_W_PACKED)
    assert base > 2048 * 75 * 16
    # without a pre-packed projection the tensor-core shape packs W2 into the workspace
    packed = ds.packed_projection_bytes(256, 151936)
    assert packed == 4 * ((151936 + 63) // 64) * 8192
    assert ds.draft_workspace_bytes(2048, 7, 151936, 256, ds.BF16, 0) >= base + packed
    assert ds.draft_workspace_bytes(2048, 7, 151936, 256, ds.BF16, ds.FLAG_FORCE_SIMT) == base
    assert ds.draft_workspace_bytes(2048, 7, 151936, 256, ds.F32, 0) == base
    assert ds.packed_projection_bytes(100, 151936) == 0 and ds.packed_projection_bytes(256, 1003) == 0
    assert ds.packed_projection_bytes(320, 1024) == 0
    assert ds.schedule_workspace_bytes(2048, 7) >= 2048 * 7 * 24
    assert ds.verify_workspace_bytes(64, 151936) > 0
    assert lib.dspark_draft_workspace_bytes(ds.Dims(0, 7, 10, 16, ds.F32, 0)) == 0


def test_host_validation_needs_no_device(lib):
    # argument errors are reported before any CUDA call
    import speculative_decoding_draft_gb300 as ds
    dims = ds.Dims(4, 7, 1000, 16, ds.F32, 0)
    null = None
    assert lib.dspark_draft_markov_sample(null, null, null, null, null, null, 0, dims, null, null, null, null, null,
                                          0, null, null) == 1
    one = ctypes.c_void_p(256)
    bad = ds.Dims(4, 17, 1000, 16, ds.F32, 0)
    assert lib.dspark_draft_markov_sample(one, one, one, one, one, one, 0, bad, one, null, null, null, one, 1 << 20,
                                          one, null) == 2
    bad = ds.Dims(4, 7, 1000, 16, 7, 0)
    assert lib.dspark_draft_markov_sample(one, one, one, one, one, one, 0, bad, one, null, null, null, one, 1 << 20,
                                          one, null) == 3
    # packing: null pointers, unsupported shapes and dtypes, short output
    pdims = ds.Dims(1, 1, 1024, 256, ds.BF16, 0)
    assert lib.dspark_draft_pack_projection(null, pdims, one, 1 << 30, null) == 1
    assert lib.dspark_draft_pack_projection(one, ds.Dims(1, 1, 1024, 96, ds.BF16, 0), one, 1 << 30, null) == 13
    assert lib.dspark_draft_pack_projection(one, ds.Dims(1, 1, 1024, 256, ds.F32, 0), one, 1 << 30, null) == 13
    assert lib.dspark_draft_pack_projection(one, pdims, one, 1024, null) == 10
    assert lib.dspark_draft_markov_sample(one, one, one, one, one, one, 0, dims, one, null, null, null, one, 16,
                                          one, null) == 10
    assert lib.dspark_schedule_survival(one, one, one, 10, 4, 0, one, one, null, null, null, one, 1 << 20, one,
                                        null) == 2
    # RNN head: null cell inputs, a packed projection, the workspace query
    rd = ds.Dims(4, 7, 1000, 16, ds.F32, 0)
    assert lib.dspark_draft_rnn_sample(one, one, one, null, one, one, one, one, 0, rd, one, null, null, null, one,
                                       1 << 20, one, null) == 1
    assert lib.dspark_draft_rnn_sample(one, one, one, one, one, one, one, one, 0,
                                       ds.Dims(4, 7, 1000, 16, ds.BF16, ds.FLAG_W_PACKED), one, null, null, null,
                                       one, 1 << 20, one, null) == 13
    assert lib.dspark_draft_rnn_workspace_bytes(rd) >= lib.dspark_draft_workspace_bytes(rd) + 2 * 4 * 4 * 16
    assert lib.dspark_draft_rnn_workspace_bytes(ds.Dims(4, 7, 1000, 16, ds.BF16, ds.FLAG_W_PACKED)) == 0
    # scheduler variants
    assert lib.dspark_schedule_capacity(one, one, one, 10, 4, 7, null, null, null, null, one, 1 << 20, one,
                                        null) == 1
    assert lib.dspark_schedule_capacity(one, one, one, 10, 4, 7, one, null, one, null, one, 1 << 20, one,
                                        null) == 1                      # ell without tgt_off
    assert lib.dspark_schedule_capacity(one, one, one, 10, 4, 7, one, null, null, null, one, 16, one, null) == 10
    assert lib.dspark_schedule_topk(one, one, null, 4, 7, one, one, null, null, one, 1 << 20, one, null) == 1
    assert lib.dspark_schedule_topk(one, one, one, 4, 17, one, one, null, null, one, 1 << 20, one, null) == 2
    assert lib.dspark_schedule_threshold(one, one, 0.5, 2, 4, 7, one, one, null, null, one, null) == 2
    assert lib.dspark_schedule_threshold(one, one, float("nan"), 0, 4, 7, one, one, null, null, one, null) == 9
    vd = ds.Dims(4, 7, 1000, 0, ds.BF16, 0)
    assert lib.dspark_verify_ragged(one, null, one, one, one, one, one, 0, vd, one, one, ctypes.c_void_p(300),
                                    1 << 30, one, null) == 10


def test_verify_markov_host_validation(lib):
    # the recompute verification: null pointers, shapes without a tensor-core path, short workspaces
    import speculative_decoding_draft_gb300 as ds
    one = ctypes.c_void_p(256)
    null = None
    dims = ds.Dims(4, 7, 1024, 256, ds.BF16, ds.FLAG_W_PACKED)
    args = [one] * 11
    assert lib.dspark_verify_markov(*([null] + args[1:]), 0, dims, one, one, one, 1 << 30, one, null) == 1
    assert lib.dspark_verify_markov_workspace_bytes(dims) > lib.dspark_verify_workspace_bytes(4, 1024)
    assert lib.dspark_verify_markov_workspace_bytes(ds.Dims(4, 7, 1024, 256, ds.F32, 0)) == 0
    assert lib.dspark_verify_markov_workspace_bytes(ds.Dims(4, 7, 1024, 96, ds.BF16, 0)) == 0
    assert lib.dspark_verify_markov(*args, 0, ds.Dims(4, 7, 1024, 96, ds.BF16, 0), one, one, one, 1 << 30, one,
                                    null) == 13
    assert lib.dspark_verify_markov(*args, 0, dims, one, one, one, 16, one, null) == 10
    # a W given as is is packed into the workspace, which grows by the packed size
    unpacked = ds.Dims(4, 7, 1024, 256, ds.BF16, 0)
    assert (lib.dspark_verify_markov_workspace_bytes(unpacked) - lib.dspark_verify_markov_workspace_bytes(dims)
            >= lib.dspark_draft_packed_projection_bytes(256, 1024))
