"""The bounds-checking build against the small-shape parity suites.

A library built with CONVF_DEBUG_BOUNDS checks every hand-computed global index of its kernels
against the tensor the launch parameters describe, skips an access that falls outside and reports
CONVF_ERR_BOUNDS through the handle's status word.  The small-shape cases of the GPU suites run
here in a child process that loads that build (CONVF_DEBUG_BOUNDS=1): every kernel variant, tile
width, epilogue mode and edge case they cover must still match the oracle and end with status
CONVF_OK, so no index of theirs ever left its tensor.  (The build reports rather than faults: a
violation skips the access, so the run stays safe for the GPU.)
"""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

# the small cases of each suite (whole outputs against the oracle, status checked after each run)
SELECTION = [
    ("test_gpu_parity.py", "single_conv or small_shapes or window_variant or depthwise_every or "
                           "both_activation or every_tile_width or halo or stream_k or kblocks or "
                           "activations or int8_bit_exact or zero_point or forced_through or non_default or "
                           "back_to_back"),
    ("test_gpu_epilogue.py", "every_output or inplace or halo_and_depthwise"),
    ("test_gpu_int8.py", "bit_exact or tile_widths or largest_chunk or mma_sync or zero_points_matter"),
    ("test_gpu_grouped.py", "every_output or tile_widths or residual_and_bf16"),
    ("test_gpu_preact.py", "every_output"),
    ("test_gpu_mbblock.py", "every_output"),
]


def test_small_suites_under_the_bounds_checking_build():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, CONVF_DEBUG_BOUNDS="1")
    # build the bounds-checking library first (its own object folder), then run the suites
    subprocess.run([sys.executable, "-c", "from convolution_onnx_conv_gb300 import _build; "
                    "_build.build(debug_bounds=True)"], cwd=ROOT, env=env, check=True)
    # the child processes load that build, not the ordinary one
    probe = subprocess.run([sys.executable, "-c", "import convolution_onnx_conv_gb300 as cf; cf.load_library(); "
                            "print(cf.library_path())"], cwd=ROOT, env=env, capture_output=True, text=True, check=True)
    assert probe.stdout.strip().endswith("libconvfused_bounds.so"), probe.stdout
    for fname, expr in SELECTION:
        res = subprocess.run([sys.executable, "-m", "pytest", os.path.join("tests", fname), "-m", "gpu", "-q",
                              "-x", "-p", "no:cacheprovider", "-k", expr], cwd=ROOT, env=env,
                             capture_output=True, text=True)
        tail = (res.stdout + res.stderr)[-3000:]
        assert res.returncode == 0, f"{fname} under the bounds-checking build:\n{tail}"
        assert " passed" in res.stdout and "deselected" in res.stdout, tail
