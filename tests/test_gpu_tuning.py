"""The attention kernel under non-default tuning (fewer warps, shallow rings,
two CTAs per SM, no fine-grained tail, other split and piece sizes), each in a child
process because the tuning variables are read once per process."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CONFIGS = {
    "4warps_2stages_2ctas": {"PA_DECODE_WARPS": "4", "PA_DECODE_MAX_STAGES": "2",
                             "PA_DECODE_CTAS_PER_SM": "2"},
    "1stage": {"PA_DECODE_MAX_STAGES": "1"},
    "no_tail_split16": {"PA_DECODE_TAIL_WAVES": "0", "PA_DECODE_SPLIT_BLOCKS": "16"},
    "wide_tail_split24": {"PA_DECODE_TAIL_WAVES": "6", "PA_DECODE_SPLIT_BLOCKS": "24"},
    "tiny_pieces": {"PA_DECODE_TAIL_WAVES": "8", "PA_DECODE_PIECE_BLOCKS": "1"},
}


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_parity_under_tuning(gpu, name):
    env = dict(os.environ)
    env.update(CONFIGS[name])
    r = subprocess.run([sys.executable, "-m", "tests.tuned_child"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]


@pytest.mark.parametrize("tc", ["0", "1"], ids=["mma_sync", "tcgen05"])
def test_prefill_parity_per_kernel(gpu, tc):
    """Chunked prefill through each of its two tensor-core kernels."""
    env = dict(os.environ, PA_PREFILL_TC=tc)
    r = subprocess.run([sys.executable, "-m", "tests.prefill_child"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]


@pytest.mark.parametrize("impl", ["phases", "grouped"])
def test_cascade_implementations(gpu, impl):
    """The shared- and grouped-prefix entry points each on one cascade
    implementation (PA_CASCADE, read once per process): the three phases
    (prefix phase on the chunked-prefill kernels, suffix decode, combine) or
    the grouped decode (one attention launch over shared and own units, which
    also merges each sequence's splits).  By default the grouped entry points use the grouped
    decode and the single-prefix ones the phases; both pass the same tests."""
    env = dict(os.environ, PA_CASCADE=impl)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p",
                        "no:cacheprovider", "tests/test_gpu_shared_prefix.py",
                        "tests/test_gpu_grouped_prefix.py", "tests/test_gpu_grouped_random.py"],
                       cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
