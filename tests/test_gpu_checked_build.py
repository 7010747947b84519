"""The checked build (libspl_checked.so) on the small and ragged parity cases.

In the checked build every shared- and global-memory index of the kernels is tested before the
access; a bad index is recorded in a device debug array (and the access skipped), nothing traps.
These tests switch the binding to that build, run the parity cases of the other test files
through it (each still compares with the oracle bit for bit), and then require that no check
failed.  They also read the sender's select-path counters, which must account for every chunk.
"""
import pytest
import torch

import compressed_pseudo_gradient_gb300 as spl

import test_gpu_codec_variants as variants
import test_gpu_parity as parity
import test_gpu_sharded as sharded_cases

pytestmark = pytest.mark.gpu


@pytest.fixture()
def checked():
    torch.cuda.synchronize()
    prev = spl.use_library(spl.checked_library_path())
    spl.debug_words(reset=True)
    try:
        yield
    finally:
        torch.cuda.synchronize()
        spl.use_library(prev)


def assert_clean(what):
    torch.cuda.synchronize()
    d = spl.debug_words(reset=True)
    assert d["failures"] == 0 and d["sites"] == 0, f"{what}: failed checks {d}"
    paths = d["whole"] + d["rank32"] + d["rank64"] + d["generic"]
    assert paths == d["chunks"], f"{what}: select paths do not add up: {d}"
    return d


def test_checked_build_is_the_one_loaded(checked):
    lib = spl.library()
    assert hasattr(lib, "spl_debug_read")
    assert spl.library_path() == spl.checked_library_path()


def test_sender_cases_touch_nothing_out_of_bounds(checked):
    parity.test_tiny_workload_all_chunks()
    for n in (1, 63, 4095, 4097, 3 * 4096 + 1, 40 * 4096 + 123):
        for dtype in (torch.float32, torch.bfloat16):
            parity.test_edge_sizes(n, dtype)
    parity.test_degenerate_chunks()
    parity.test_select_window_edges()
    parity.test_bf16_ties_stress()
    parity.test_exact_ties_in_the_boundary_bin_and_sparse_chunks()
    parity.test_nonfinite_inputs_flagged_and_deterministic()
    parity.test_heavy_tail_bf16_medium_all_chunks()
    parity.test_decoder_layer_multi_tensor_small_all_chunks()
    parity.test_multi_tensor_matches_single_calls_and_splits_long_tables()
    d = assert_clean("sender cases")
    # the planted cases reach every select path
    for path in ("whole", "rank32", "rank64", "full_scan", "generic"):
        assert d[path] > 0, f"path {path} not reached: {d}"


def test_host_error_buffer_and_streams_touch_nothing_out_of_bounds(checked):
    for dtype in (torch.float32, torch.bfloat16):
        parity.test_error_buffer_in_pinned_host_memory(dtype)
    parity.test_multi_tensor_host_error_buffers()
    parity.test_resume_from_host_copy_of_error_buffer()
    parity.test_side_stream_and_stream_order()
    assert_clean("host error buffer")


def test_receiver_cases_touch_nothing_out_of_bounds(checked):
    parity.test_pack_unpack_match_oracle()
    parity.test_malformed_records_rejected_like_oracle(False)
    parity.test_malformed_records_rejected_like_oracle(True)
    for P in (1, 5, 8, 24):
        parity.test_decode_without_validation_matches_oracle(P)
    parity.test_peer_stats_match_oracle()
    parity.test_many_peers_span_several_groups(65)
    parity.test_many_peers_span_several_groups(256)
    assert_clean("receiver cases")


def test_sharded_slices_touch_nothing_out_of_bounds(checked):
    sharded_cases.test_slices_compress_and_decode_like_the_whole_tensor(
        3, 37 * 4096, torch.bfloat16)
    sharded_cases.test_slices_compress_and_decode_like_the_whole_tensor(
        4, 2 * 4096 + 5, torch.float32)
    assert_clean("sharded slices")


@pytest.mark.parametrize("codec", variants.CODECS)
def test_codec_variants_touch_nothing_out_of_bounds(checked, codec):
    for dtype in (torch.float32, torch.bfloat16):
        variants.test_variant_rounds_match_oracle(codec, dtype)
        variants.test_variant_exact_ties_and_sparse_chunks(codec, dtype)
    variants.test_variant_edge_chunks(codec)
    variants.test_variant_nonfinite_inputs_flagged_and_deterministic(codec)
    if codec[2] == variants.MAX:
        variants.test_variant_decode_matches_oracle(codec)
        variants.test_variant_many_peers_span_several_groups(codec, 70)
    assert_clean(f"codec {codec}")
