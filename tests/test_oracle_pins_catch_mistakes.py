"""The oracle's pins catch plausible mistakes in the oracle.

For every entry of ``tests/_plants.py`` (a dropped term, a wrong sign, bias,
index or comparison, a transposed operand, a swapped byte or nibble order),
a child pytest process installs that one mistake in the oracle and runs the
pin module that covers the function. The pins must fail there. A control
child with no mistake must pass, so a failure is the plant's doing. The
children run on the CPU, several at a time.
"""

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

from tests import _plants

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CONTROL = "no mistake"


def _run_child(plant: str, module: str):
    env = dict(os.environ)
    env.pop("MJ_PLANT", None)
    if plant != CONTROL:
        env["MJ_PLANT"] = plant
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "not gpu",
           os.path.join("tests", module)]
    r = subprocess.run(cmd, cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True,
                       timeout=600)
    return r.returncode, r.stdout[-3000:]


@pytest.fixture(scope="module")
def outcomes():
    jobs = [(name, module) for name, (_, module) in _plants.PLANTS.items()]
    jobs += [(CONTROL, m) for m in sorted({m for _, m in jobs})]
    with ThreadPoolExecutor(max_workers=max(2, min(8, os.cpu_count() or 2))) as ex:
        futs = {(name, module): ex.submit(_run_child, name, module) for name, module in jobs}
        return {key: f.result() for key, f in futs.items()}


@pytest.mark.parametrize("module", sorted({m for _, m in _plants.PLANTS.values()}))
def test_pins_pass_without_a_planted_mistake(outcomes, module):
    rc, out = outcomes[(CONTROL, module)]
    assert rc == 0, out


@pytest.mark.parametrize("plant", list(_plants.PLANTS))
def test_planted_mistake_fails_a_pin(outcomes, plant):
    module = _plants.PLANTS[plant][1]
    rc, out = outcomes[(plant, module)]
    # pytest exits 1 when a test failed; anything else (0: the mistake went
    # unnoticed; 2-4: the run itself broke) does not count as a pin catching it
    assert rc == 1 and " failed" in out, f"{plant} not caught by {module} (exit {rc}):\n{out}"
