"""CPU oracle for the AWQ scale search (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never uses it.
"""
from .awq_oracle import (  # noqa: F401
    alpha_grid,
    channel_magnitude,
    dequantize_scaled,
    first_argmin,
    fold_inverse_scale,
    layer_loss,
    output_error_rows,
    pack_codes,
    packed_words,
    quantize_groups,
    scale_vector,
    search,
    unpack_codes,
    w4a16_matvec,
)
