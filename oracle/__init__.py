"""CPU oracle for the top-k MoE layer (test infrastructure only).

Only the tests, `__graft_entry__.smoke()` and the bench's CPU-baseline leg may
import this package.  The product path (`combine_moe_gate_gb300`) never does,
and nothing here imports the product package: the two share only the seeded
input generators in `synth`.

`moe_oracle.c` holds the sparse, loop-level restatement of the method; `dense`
holds the dense one-hot-mask / einsum formulation the pages describe, used to
pin the sparse loops.  Every function cites the passage it follows.
"""

from .core import (  # noqa: F401
    ACT,
    build,
    capacity,
    decode,
    decode_bwd,
    encode,
    encode_bwd,
    fc_fp8,
    ffn_bwd,
    ffn_rows,
    fp8_decode,
    fp8_encode,
    gate_bwd,
    gate_chunk,
    gate_logits,
    gates,
    get_threads,
    kept_rows,
    layer_backward,
    layer_forward,
    locations,
    quantize_rows_fp8,
    round_bf16,
    set_threads,
    to_f32,
    topk,
)
