"""CPU oracle for the quantized-KV speculative decode-attention path.

TEST INFRASTRUCTURE ONLY.  The library's product path never imports, calls or
links anything here.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg do.  See ``kvq_oracle`` for what each function
computes and which passage of the pages it follows.
"""
from .kvq_oracle import (  # noqa: F401
    FORMAT_BITS,
    CENTER_SHIFT,
    MID_NIBBLE,
    MODES,
    SLAB,
    OracleCache,
    all_scores,
    attend,
    gather_selected,
    mode_codes_scale,
    mode_zero,
    pack_k_plane,
    pack_v_plane,
    quantize_key_group,
    quantize_minmax,
    quantize_value_group,
    score_group,
    split_hierarchical,
    summed_query,
    topk,
)
