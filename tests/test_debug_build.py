"""The bounds-checking build (libspecdec_debug.so, the sources compiled with
-DSPEC_DEBUG): every kernel tests the indices that depend on its inputs
against their buffers, skips an access that falls outside and counts it.
With no memory checker on the GPU, this runs the GPU parity suite's small
and adversarial cases (ragged vocabularies, NaN and empty rows, trees from 4
to 64 nodes, retrieve links that loop, forced fallbacks, the chain verify,
TLI maps with gaps, the pruned head's ragged tiles, filtering, the captured
step) against that build in a child process; conftest's fixture asserts
that each test met no out-of-range index, and this test that the child ran
them and passed."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_release_library_has_no_count():
    sd = pytest.importorskip("speculative_decoding_draft_select_gb300")
    if sd.library_path.endswith("libspecdec_debug.so"):
        pytest.skip("running under the debug build")
    if not os.path.exists(sd.library_path):
        pytest.skip("library not built")
    with pytest.raises(sd.SpecError) as e:
        sd.spec_debug_bounds()
    assert e.value.rc == -2


@pytest.mark.gpu
@pytest.mark.timeout(1800)
def test_parity_suite_under_the_bounds_checking_build():
    if os.environ.get("SPECDEC_DEBUG") == "1":
        pytest.skip("already inside the debug run")
    from speculative_decoding_draft_select_gb300.build import build
    lib = build(debug=True)
    assert lib.endswith("libspecdec_debug.so") and os.path.exists(lib)
    env = dict(os.environ, SPECDEC_DEBUG="1")
    # the full-size cases repeat the small ones' code paths at bench sizes
    cmd = [sys.executable, "-m", "pytest", "tests/test_gpu_parity.py", "tests/test_zz_no_alloc.py", "-m", "gpu",
           "-k", "not full_size", "-q", "-p", "no:cacheprovider"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1700)
    tail = (r.stdout + r.stderr)[-4000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and " error" not in r.stdout, tail
