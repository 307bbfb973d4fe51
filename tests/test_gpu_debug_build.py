"""The debug build (device-side bounds checks) on the GPU.

`build.py --debug` compiles libparallax_attn_debug.so with -DPARALLAX_DEBUG_CHECKS: before
each global write and bulk copy they cover, the kernels check that the element range lies
inside its tensor, and a failed check raises DEVERR_BOUNDS in the device error word instead
of touching memory outside the tensor.  This test runs the canary tests (every entry point on
odd shapes, guard bands around every output and workspace, and a device-error check after
each call), the failure-path tests and the small-shape parity tests of the decode and the
prefill against the oracle in a child process that loads the debug library; every one must
pass with no error bit set.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_library_passes_the_checked_suite():
    from softmax_covariance_correction_pass_b300 import build as pxbuild

    pxbuild.build(debug=True)
    env = dict(os.environ, PARALLAX_LIBRARY="debug")
    probe = subprocess.run(
        [sys.executable, "-c", "import softmax_covariance_correction_pass_b300 as px; "
         "print(px.LIB_PATH, px.parallax_debug_checks())"],
        env=env, cwd=os.path.dirname(HERE), capture_output=True, text=True, timeout=300)
    assert probe.returncode == 0, probe.stderr
    assert probe.stdout.split()[-2].endswith("libparallax_attn_debug.so")
    assert probe.stdout.split()[-1] == "True"
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           os.path.join(HERE, "test_gpu_canaries.py"), os.path.join(HERE, "test_gpu_failure.py"),
           os.path.join(HERE, "test_gpu_decode.py") + "::test_bf16_small",
           os.path.join(HERE, "test_gpu_decode.py") + "::test_f32_small",
           os.path.join(HERE, "test_gpu_prefill.py") + "::test_bf16_shapes"]
    r = subprocess.run(cmd, env=env, cwd=os.path.dirname(HERE), capture_output=True, text=True,
                       timeout=1500)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout, tail
