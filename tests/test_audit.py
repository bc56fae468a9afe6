"""Source audits of the product path.

* No atomics anywhere in the CUDA sources: each output tile is owned by one
  CTA over the whole K, so nothing accumulates across CTAs (the pages'
  backward-contract audit forbids atomicAdd).
* No multi-GPU multicast (multimem / NVLS), no TMA multicast load
  (cp.async.bulk ... .multicast::cluster): the library runs as one replica
  per GPU, and every operand byte reaches shared memory through a plain load.
  The one multicast form allowed is the MMA commit that signals both CTAs of
  a pair (tcgen05.commit ... .multicast::cluster), an mbarrier arrive, not a
  copy.  No Triton, no torch.compile on the product path.
* The product path never imports the oracle, and the oracle never imports
  the product path.
"""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "weight_grad_gemm_gb300")


def files(top, exts):
    for d, _, fs in os.walk(top):
        if "_build" in d or "__pycache__" in d:
            continue
        for f in fs:
            if f.endswith(exts):
                yield os.path.join(d, f)


def strip_comments(text):
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.sub(r"//[^\n]*", "", text)


def test_no_atomics_in_cuda_sources():
    pat = re.compile(r"\batomic[A-Z]\w*\s*\(|\batom\.|\bred\.|\bmultimem\.")
    hits = []
    for f in files(os.path.join(PKG, "csrc"), (".cu", ".cuh", ".h")):
        code = strip_comments(open(f).read())
        for m in pat.finditer(code):
            hits.append((os.path.basename(f), m.group(0)))
    assert not hits, hits


def test_no_multigpu_multicast_triton_or_compile():
    for f in files(PKG, (".cu", ".cuh", ".py")):
        code = open(f).read()
        assert "multimem" not in code, f
        assert not re.search(r"^\s*(import|from)\s+triton", code, re.M), f
        assert "torch.compile" not in code, f


def test_no_tma_multicast_loads():
    """Every PTX string that names .multicast::cluster must be a tcgen05
    commit, never a bulk copy."""
    hits = []
    for f in files(os.path.join(PKG, "csrc"), (".cu", ".cuh", ".h")):
        code = strip_comments(open(f).read())
        # join adjacent string literals so one instruction is one string
        joined = re.sub(r'"\s*\n\s*"', "", code)
        for lit in re.findall(r'"([^"\n]*)"', joined):
            if "multicast" in lit and "tcgen05.commit" not in lit:
                hits.append((os.path.basename(f), lit.strip()[:80]))
            if re.search(r"cp\.async\.bulk[^;]*multicast", lit):
                hits.append((os.path.basename(f), lit.strip()[:80]))
    assert not hits, hits


def test_kernel_form_choice_has_no_multicast_form():
    api = open(os.path.join(PKG, "csrc", "forge_api.cu")).read()
    assert '"quad"' not in api
    assert "NPAIR" not in open(os.path.join(PKG, "csrc", "forge_kernel.cuh")).read()


def test_product_and_oracle_are_separate():
    for f in files(PKG, (".py", ".cu", ".cuh")):
        code = open(f).read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", code, re.M), f
        assert "forge_oracle" not in code, f
    for f in files(os.path.join(ROOT, "oracle"), (".py", ".c")):
        code = open(f).read()
        assert "weight_grad_gemm_gb300" not in code, f
        assert "forge_kernel" not in code and "forge.h" not in code, f


def test_no_closed_batch_copy_calls():
    names = ["cudaMemcpyBatch" + "Async", "cudaMemcpy3DBatch" + "Async",
             "cuMemcpyBatch" + "Async", "cuMemcpy3DBatch" + "Async"]
    for top in (PKG, os.path.join(ROOT, "tests"), os.path.join(ROOT, "oracle")):
        for f in files(top, (".py", ".cu", ".cuh", ".c", ".h")):
            code = open(f).read()
            for n in names:
                assert n not in code, (f, n)
