"""CPU oracle for the batched speculative-decoding verify step (float64).

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, independent
restatement of what the verify step computes, used to check the CUDA path.  It
shares no code with the CUDA library or its Python binding and imports
neither.  Only tests/, the smoke check and the bench's CPU-baseline (and
reference-arm) leg may import it; the product path never does.

Modules (each cites the passages it follows):
  philox     Philox4x32-10 and the verify uniforms
  sampling   processing (temperature, nucleus), accept rule, residual / bonus
             draw, batch loop, near-tie audit
  attention  ragged verify attention (plus the shared-prefix arrangement)
  append     ragged append of accepted K/V rows
  step       the three composed
  draft      the draft side: draft-token draw (Philox stream 1) and one draft
             position (single-row attention, append, draw)
"""
from .philox import philox4x32, verify_uniforms, word_to_uniform
from .sampling import (process_row, accept, residual, sample_index, verify_sequence,
                       reject_sample, to_f64, bf16_bits_to_f64, TIE_EPS, TIE_ACCEPT, TIE_DRAW,
                       DEV_CAPACITY, DEV_BAD_TOKEN, DEV_NONFINITE, DEV_EMPTY_RESIDUAL,
                       DEV_BAD_LENGTH, DEV_BAD_PARAM, params_ok)
from .attention import attention_row, verify_attention
from .append import kv_append
from .step import verify_step
from .draft import draft_sample, draft_step
