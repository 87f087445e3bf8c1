"""CPU oracle for ring attention (test infrastructure, not product code).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import or execute anything in this package.  It shares no
code with the CUDA path; the only common piece is the ``ragen`` input
generator, which holds no attention arithmetic.

Everything here is plain NumPy in float64: inputs (bf16 or fp32) are upcast
exactly, so the oracle computes the mathematical result of the method on the
given inputs, up to float64 rounding.

Sources (the pages these functions follow):
  * "Ring Attention" glossary page (ultralytics.com), section "Como funciona a
    atencao em anel": N blocks, device i keeps query block i, at step s it
    holds key/value block j = (i - s) mod N received from the previous
    device; accumulated exponentiated scores and weighted values divided at
    the end; production kernels subtract a running maximum; causal masking
    and Striped Attention (tokens spread evenly over devices).
  * "Sequence parallelism and ring attention" pages (aiunderstanding.org),
    sections "Immersione profonda" / "Approfondimento tecnico": contiguous
    token blocks, online softmax with a running max and running normaliser,
    earlier partial sums rescaled when a larger score arrives, result
    mathematically identical to full attention.
  * "Ring Attention la gi?" (thienlv.com), section "Uu Diem": compatible with
    GQA.
  * Training as the use (Italian aiunderstanding.org page, "Implementazione
    nel mondo reale"; glossary page, training throughput and
    context_parallel): the gradients are the chain rule of the plain
    definition; the ring-order backward is this oracle's reading.

Pin status: every function here is pinned by a CPU test against something
other than itself (brute force, closed forms, a library routine, the pages'
worked example); see ``tests/test_oracle.py``.
"""
from .attention import (  # noqa: F401
    bf16_bits_to_f64,
    positions,
    stripe_perm,
    to_token_order,
    to_shard_major,
    attend_rows,
    full_attention,
    ring_attention,
    merge,
    fold_schedule,
    toy_ring_no_max,
    ulysses_exchange,
    attention_backward,
    attention_backward_rows,
    attention_backward_key_rows,
    backward_uniform_scores,
    ring_attention_backward,
    ring_step_backward_block,
)
