"""The bounds-checking build (libwsattn_debug.so, compiled with WSATTN_DEBUG):
its kernels check every TMA coordinate, tensor-memory column range,
shared-memory layout, output row and work-item index before the access and
report a failed check through the device status word (no trap).  This stands
in for a memory checker.

test_kernels_pass_bounds_checks reruns a set of the parity tests in a child
process that loads the debug library (WSATTN_LIBRARY): tiny and small, the
edge shapes, block sizes, degenerate inputs, every mask variant, window
bounds and the pre-attention producer.  Each of those tests already requires
device status 0 after its kernels and outputs within the parity bar, so a
failed bounds check fails the run.  test_library_is_debug_build runs only in
that child and confirms which library it loaded.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
IN_CHILD = os.environ.get("WSATTN_EXPECT_DEBUG") == "1"

RERUN = [
    "tests/test_gpu_forward.py::test_forward_full_parity",
    "tests/test_gpu_forward.py::test_edge_shapes_full_parity",
    "tests/test_gpu_forward.py::test_merged_tails_ignore_keys_outside_the_row_frame",
    "tests/test_gpu_forward.py::test_block_sizes_tiny",
    "tests/test_gpu_forward.py::test_block_sizes_dense_frame_span",
    "tests/test_gpu_forward.py::test_block_sizes_step_buffers",
    "tests/test_gpu_forward.py::test_degenerate_inputs",
    "tests/test_gpu_forward.py::test_batch_mismatch_and_status",
    "tests/test_gpu_mask_variants.py::test_variant_forward_full_parity",
    "tests/test_gpu_mask_variants.py::test_random_shapes_full_parity",
    "tests/test_gpu_mask_variants.py::test_variant_forward_online_and_d64",
    "tests/test_gpu_mask_variants.py::test_variant_window_bounds",
    "tests/test_gpu_window_bound.py::test_window_bound_flips_eligibility_and_forward_matches",
    "tests/test_gpu_prepare.py::test_prepare_matches_oracle",
    "tests/test_gpu_produce.py::test_produce_full_parity",
    "tests/test_gpu_zy_debug_build.py::test_library_is_debug_build",
]


@pytest.mark.skipif(IN_CHILD, reason="runs in the parent process only")
def test_kernels_pass_bounds_checks():
    import frame_aligned_window_gb300 as fw
    lib = fw.DEBUG_LIB_PATH
    assert os.path.exists(lib), "build it with `python frame_aligned_window_gb300/build.py --debug`"
    env = dict(os.environ, WSATTN_LIBRARY=lib, WSATTN_EXPECT_DEBUG="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           *RERUN]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0, (r.stdout[-4000:], r.stderr[-2000:])
    assert " passed" in r.stdout and "skipped" not in r.stdout.splitlines()[-1], r.stdout[-500:]


@pytest.mark.skipif(not IN_CHILD, reason="runs only in the child process of the test above")
def test_library_is_debug_build():
    import frame_aligned_window_gb300 as fw
    assert os.path.samefile(fw.LIB_PATH, fw.DEBUG_LIB_PATH)
    assert fw.wsattn_build_flags() & fw.BUILD_DEBUG
