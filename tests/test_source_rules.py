"""Rules on the CUDA sources, checked as text (no GPU, no build).

* No bulk or tensor copy (cp.async.bulk, cp.async.bulk.tensor) carries
  .multicast::cluster.  The kernels here load every tile into the shared memory
  of the CTA that uses it; a multicast load would write other CTAs' shared
  memory, which these kernels never set up for.  The MMA thread's commit to the
  stage barriers of both CTAs of a pair (tcgen05.commit ... multicast::cluster)
  is an mbarrier arrive, not a load, and stays allowed.
* No kernel stops itself with a trap: a wait that gives up records a status
  word and returns.
"""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "dense_fp16_tensor_gemm_gb300", "csrc")


def _sources():
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(CSRC, name)) as f:
                yield name, f.read()


def _strings(text):
    """The string literals of a C++ source (inline PTX lives in them), with
    adjacent literals joined the way the compiler joins them."""
    text = re.sub(r"//[^\n]*", "", text)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    joined = re.sub(r'"\s*\n\s*"', "", text)
    return re.findall(r'"((?:[^"\\\n]|\\.)*)"', joined)


def test_sources_are_found():
    names = [n for n, _ in _sources()]
    assert "tc05_pair.cu" in names and "ptx.cuh" in names


def test_no_multicast_bulk_loads():
    bad = []
    for name, text in _sources():
        for s in _strings(text):
            if "cp.async.bulk" in s and "multicast" in s:
                bad.append((name, s))
    assert not bad, bad


def test_the_lint_sees_inline_ptx():
    """The checker finds the commit-arrive multicast the pair kernel uses, and
    the tensor loads, so an added multicast load would be seen."""
    strings = [s for _, text in _sources() for s in _strings(text)]
    assert any("tcgen05.commit" in s and "multicast::cluster" in s for s in strings)
    assert any(s.startswith("cp.async.bulk.tensor") for s in strings)
    planted = 'asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"\n' \
              '             ".multicast::cluster [%0], [%1, {%2, %3}], [%4], %5;" :: ...);'
    assert any("cp.async.bulk" in s and "multicast" in s for s in _strings(planted))


def test_no_traps():
    for name, text in _sources():
        code = re.sub(r"//[^\n]*", "", text)
        code = re.sub(r"/\*.*?\*/", "", code, flags=re.S)
        assert "__trap" not in code, name
        assert not any(re.match(r"\s*trap\s*;", s) for s in _strings(code)), name
