"""Source check of the overlapped-launch contract (csrc/pdl.cuh).

A kernel launched with programmatic stream serialisation may start while the
kernel before it in the stream is still running; it is correct only if its
first statement waits for that kernel (griddep_wait()). This test reads the
CUDA sources, finds every kernel passed to launch_pdl and checks that the body
of its definition begins with that wait. It needs no GPU.
"""
import os
import re

import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "bit_quantized_expert_softmax_b300", "csrc")


def _sources():
    out = {}
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(CSRC, name)) as fh:
                out[name] = fh.read()
    return out


def _pdl_kernels(srcs):
    names = set()
    for text in srcs.values():
        for m in re.finditer(r"launch_pdl\(\s*([A-Za-z_]\w*)", text):
            if m.group(1) not in ("void", "kernel"):   # the helper's own definition
                names.add(m.group(1))
    return sorted(names)


def _first_statement(text, kernel):
    """The first statement of the body of `__global__ ... kernel(...)`."""
    m = re.search(r"__global__\s+void[^;{]*?\b" + re.escape(kernel) + r"\s*\(", text)
    if m is None:
        return None
    i = m.end()
    depth = 1
    while depth:                     # the parameter list
        depth += {"(": 1, ")": -1}.get(text[i], 0)
        i += 1
    body = text.index("{", i) + 1
    rest = text[body:]
    rest = re.sub(r"^\s*(//[^\n]*\n\s*)*", "", rest)   # leading comments
    return rest.split(";", 1)[0].strip() + ";"


def test_every_overlapped_kernel_waits_first():
    srcs = _sources()
    kernels = _pdl_kernels(srcs)
    # the chains this build launches this way (a guard against the regex
    # silently finding nothing)
    for expected in ("fp4_gemm_kernel", "fp4_gemm_resa_kernel", "quant_x_kernel", "quant_h_kernel",
                     "combine_kernel", "router_small_kernel", "token_rank_kernel", "router_umma_kernel",
                     "gateup_ring_kernel", "down_ring_kernel", "head_gemv_kernel", "head_sample_kernel"):
        assert expected in kernels, expected
    for k in kernels:
        found = [(name, _first_statement(text, k)) for name, text in srcs.items()
                 if _first_statement(text, k) is not None]
        assert found, f"no definition of {k}"
        for name, stmt in found:
            assert stmt == "griddep_wait();", f"{k} in {name} starts with {stmt!r}"


@pytest.mark.parametrize("snippet,ok", [
    ("__global__ void k(int a) {\n    griddep_wait();\n    x = 1;\n}", True),
    ("__global__ void __launch_bounds__(256) k(int a, int b) {\n    // note\n    griddep_wait();\n}", True),
    ("__global__ void k(int a) {\n    x = 1;\n    griddep_wait();\n}", False),
])
def test_first_statement_parser(snippet, ok):
    assert (_first_statement(snippet, "k") == "griddep_wait();") == ok
