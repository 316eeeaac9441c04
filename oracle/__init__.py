"""Plain float64 CPU oracle for the paged NVFP4 KV decode path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
its Python binding) may import, call or link anything in this package; only
the tests, the package's ``smoke()`` check and ``bench.py``'s CPU-baseline leg
and reference arm use it.  It shares no code, tables or constants with the
CUDA path: every function here is restated from the published definitions it
cites, written for a reader to check by eye, with no blocking, fusion or
reordering beyond what those definitions state.

Sources, cited by page title and section:

* "A 1,048,576-token context on two RTX 5090s: forking a C++ inference engine
  for tensor-parallel and YaRN" (portfolio-site-axx.pages.dev), sections
  "YaRN, and matching what vLLM actually does" and "Things that bit me".
* "ninfer-windows-tp2" README (git.onestrm.cn/ivanov84), section
  "YaRN reference and drift guard".
* "262,144 Tokens on One RTX 5090: Qwen3.8-27B with an NVFP4 KV Cache That
  Actually Works" (stondo.github.io), sections "Why NVFP4 KV changes the math"
  and "The stack, for the impatient".
* "A 1,048,576-token context on two RTX 5090s", section "Against vLLM:
  prefill loses, decode wins, and one surprise" (the comparison engine's fp8
  KV cache); the README's sections "Dual-GPU (TP2) and YaRN 1M context" and
  "Memory, per GPU" (INT8 group-64 KV).
* The published YaRN method (Peng et al., 2023, "YaRN: Efficient Context
  Window Extension of Large Language Models"), which the first page cites as
  its reference 3, for the NTK-by-parts ramp and the attention temperature.
* The OCP 8-bit floating point (E4M3FN) and OCP microscaling (E2M1) format
  definitions for the two element codecs.

Modules:
  formats    E2M1 / E4M3 / bf16 codecs.
  yarn       YaRN inverse frequencies, mscale, cos/sin tables, rope.
  nvfp4      two-level NVFP4 block quantise / dequantise.
  fp8        per-tensor FP8 (E4M3) quantise / dequantise.
  int8       INT8 group-64 quantise / dequantise (fp16 group scales).
  paged      page-pool byte layout, scatter and gather.
  attention  dense and paged attention, split-KV partials, LSE combine.
  fp4_prefill  attention with NVFP4-quantised queries (the block-scaled
             FP4 x FP4 QK^T reading of a prefill over the NVFP4 cache).

Parity status: every function is pinned by a ``-m "not gpu"`` test against a
closed form, an invariant, an exhaustive enumeration or brute force, except
agreement of the YaRN table with one particular serving stack's dump, which
is not available ("parity unpinned" for that comparison only).
"""
