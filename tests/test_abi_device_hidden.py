"""Runs test_abi.py with the GPU hidden (CUDA_VISIBLE_DEVICES="") when this
process can see one.  test_abi.py passes made-up device addresses that host
validation must refuse; with no device visible, a validation regression
returns a wrong status code instead of launching a kernel on a shared GPU."""
import os
import subprocess
import sys

import pytest

from test_abi import ROOT, gpu_visible


def test_abi_checks_run_with_the_device_hidden():
    if not gpu_visible():
        pytest.skip("no GPU visible: test_abi.py runs in this process")
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_abi.py")], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-4000:]
    assert " passed" in r.stdout and "skipped" not in r.stdout.splitlines()[-1], r.stdout[-2000:]
