"""CPU oracle for the decode quant + quantized-linear path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, deliberately
obvious restatement of what the path computes, written from the pages'
definitions.  Only the test-suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product path (the CUDA library and its Python binding) never imports,
links or executes anything here, and this package never imports the product.

Sources (page title, then section):
  [W8A8]  "DeepSeek-V4 W8A8 performance analysis: small M, NZ layout and
          measurement method" (akiyangdev llm-inference-notes).
  [PR]    "SGLang PR #34277 digest: the DSV4 FP8 quant kernel writes
          DeepGEMM's TMA-aligned packed UE8M0 scales" (prhub).
  [DF]    "Reshaping LLM inference dataflow: DeepSeek V4 950 low-precision
          optimisation retrospective" (0539edu).

Modules:
  codecs  bf16 / E4M3 / UE8M0 encodings, from the format definitions.
  int8    per-token INT8 dynamic quant, W8A8 linear, fused quant+linear.
  fp8     per-128 group FP8 quant with packed UE8M0 scales, fp32->packed
          repack, fp8 weight block quant, block-scaled grouped einsum.
  norm    RMSNorm fused with the INT8 per-token or FP8 per-group quant.
  mx      32-element block-scaled FP8 (UE8M0 scale per block) and its linear.
  moe     sort-by-expert, gather, grouped W8A8, SwiGLU+requant, combine.
  layout  load-time K-major weight repack.

Every function here is pinned by ``tests/test_oracle_*.py`` against values
fixed by the pages, closed forms, invariants or brute force.
"""
from . import codecs, int8, fp8, moe, norm, mx, layout  # noqa: F401
