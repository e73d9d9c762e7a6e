"""CPU oracle (float64 NumPy) of the folded-Hadamard ternary Packed layer.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference legs of ``bench.py``; never by the library.

Parity status of each function (what pins it is in tests/test_oracle_pins.py):
  fwht            pinned: explicit Sylvester matrix, closed forms, worked examples
  pack_w2         pinned: hand-computed words
  unpack_w2       pinned: hand-computed words, round trip
  decode_w2       pinned: value set {-s,0,s}, code counts, worked example
  packed_linear   pinned: brute-force loops, fold invariant, embedding cross-check
  embed_lookup    pinned: forward transform recovers the dequantised row
  pq2_0_*, ptq1_0_*, transcode_to_w2
                  pinned: hand-computed blocks, round trips, invalid values refused
Parity with the trained model is unpinned (no weights exist here).
"""
from .w2_hadamard import (GROUP, BITS, CODES_PER_WORD, fwht, pack_w2, unpack_w2,
                          biases_for, decode_w2, packed_linear, rotated_input,
                          abs_product_sum, embed_lookup)
from .gguf_blocks import (PQ2_0_BYTES, PTQ1_0_BYTES, pq2_0_encode, pq2_0_decode, ptq1_0_encode,
                          ptq1_0_decode, transcode_to_w2)

__all__ = ["GROUP", "BITS", "CODES_PER_WORD", "fwht", "pack_w2", "unpack_w2",
           "biases_for", "decode_w2", "packed_linear", "rotated_input",
           "abs_product_sum", "embed_lookup", "PQ2_0_BYTES", "PTQ1_0_BYTES", "pq2_0_encode",
           "pq2_0_decode", "ptq1_0_encode", "ptq1_0_decode", "transcode_to_w2"]
