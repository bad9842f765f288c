"""Plain, slow CPU oracle for TurboQuant KV-cache compression (float64 numpy).

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may use it.  It shares no code,
table or constant with the CUDA library; both sides only consume the same
seeded inputs from ``turboquant_bit_kv_gb300.workloads``.

Every function cites the page and section it restates.  Pages:

* "TurboQuant KV Cache Compression — Spec" (Foundry attention/spec.md):
  Algorithm Detail steps 1-3, As-Built Notes, Codebook Generation,
  Hadamard Transform Detail, Optimization: Fused dequant-dot.
* "TurboQuant KV Cache (turboq2 / turboq3 / turboq4)" (llama.cpp fork
  turboquant-kv-base.md): section 4 block structures and encode pipeline.
* "RotorQuant KV Cache Compression" (RotorQuant docs): The QJL Estimator
  Formula, Key Compression Workflow, Fused Kernel Logic.
* "lmcache.v1.distributed.serde.turboquant" (LMCache serde design):
  Configuration, Tensor Layout.

``oracle.ext`` holds the further block formats (norm-corrected encode, the
dense 8-in-3 packing of 3-bit codes, the 8-bit turboq8 codec),
``oracle.headdim`` the codec at head dims 64, 96 and 160 (a dense orthogonal
rotation as an input) and ``attention_causal`` the multi-token causal
attention.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, textbook tables, library routines or values printed on
the pages; none is "parity unpinned".
"""

from .signs import splitmix64, sign_diagonal
from .codebook import lloyd_max, beta_codebook, gaussian_codebook, beta_law_moments
from .rotation import hadamard, rotate, rotate_inverse
from .codec import (block_bytes, quantize, encode, pack_block, unpack_block,
                    decode, decode_rotated, fp16_rne)
from .attention import attention_dequantized, attention_rotated, attention_causal
from .qjl import qjl_encode, qjl_term2
from .serde import serde_ranges, serde_size, serialize, deserialize

__all__ = [
    "splitmix64", "sign_diagonal", "lloyd_max", "beta_codebook",
    "gaussian_codebook", "beta_law_moments", "hadamard", "rotate",
    "rotate_inverse", "block_bytes", "quantize", "encode", "pack_block",
    "unpack_block", "decode", "decode_rotated", "fp16_rne",
    "attention_dequantized", "attention_rotated", "attention_causal", "qjl_encode", "qjl_term2",
    "serde_ranges", "serde_size", "serialize", "deserialize",
]
