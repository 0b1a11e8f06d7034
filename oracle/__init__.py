"""CPU oracle for the sparse-attention indexer decode path.

TEST INFRASTRUCTURE ONLY.  This package is the slow, plain, obviously
correct statement of what the path computes, used to check the CUDA library.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  The CUDA library and its Python binding never
import it, and it never imports them: the two share no code.  Inputs come from
the seeded generator in ``sparse_attention_indexer_nvfp4_gb300.workloads``,
which the tests hand to both sides.

Modules:

* ``formats`` - E4M3 and E2M1 value tables and the E4M3 round-to-nearest-even
  saturating encoder, written from the formats' definitions.
* ``indexer`` - NVFP4 page fields and dequantisation, decode page scores,
  64-bit page keys, exact top-16, decode row assembly, the decode step, and
  the multi-token relu-weighted scorer.
* ``mxfp8`` - MXFP8 quantisation of bf16 rows (E8M0 block scales from the
  amax's bit fields, E4M3 values), the epilogue that follows sparse decode
  attention.

Pins (checked by ``tests/test_oracle_*.py`` against the pages, closed forms
and brute force, never against the CUDA path) are listed in each function's
docstring.  Parity unpinned: none of the functions; the page layout reading
("codes of all tokens, then all scales") is a convention of the pages and is
pinned by a hand-built page fixture in ``tests/golden``.
"""
