"""FP64 CPU oracle for MSA block-sparse attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the CUDA library under ``block_sparse_attention_prefill_gb300/``;
the two meet only in the seeded inputs of ``workloads.py``.

Contents
  attention()   masked softmax attention over the selected pages (C, FP64)
  k2q_csr()     page-to-query CSR by plain loops (C)
  schedule()    the work list rule, restated in Python
  combine()     log-sum-exp merge of split partials (C, FP64)
  brute_force_attention()   numpy triple loop for tiny inputs (pins the C)
  e4m3_decode() the OCP E4M3 decoding written from the format definition
  e4m3_encode() nearest-even E4M3 rounding, saturating at 448 (C)
  e2m1_decode() the OCP E2M1 (FP4) decoding from the format definition (C)
  nvfp4_to_e4m3()  NVFP4 page pool -> E4M3 page pool: code x block scale,
                rounded to E4M3 (C)

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(no function is "parity unpinned").
"""
from .oracle import (attention, brute_force_attention, combine, e2m1_decode,
                     e4m3_decode, e4m3_encode, e4m3_table, k2q_csr, max_threads,
                     nvfp4_to_e4m3, schedule)

__all__ = ["attention", "brute_force_attention", "combine", "e2m1_decode",
           "e4m3_decode", "e4m3_encode", "e4m3_table", "k2q_csr", "max_threads",
           "nvfp4_to_e4m3", "schedule"]
