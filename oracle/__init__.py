"""CPU oracle for paged GQA decode attention with per-tile LSE and an FP32 LSE merge.

TEST INFRASTRUCTURE ONLY.  This package is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the ``cpu_baseline`` / reference legs of
``bench.py``; nothing on the product path (the ``paged_decode_attention_attn_gb300``
package, its C-ABI library or its kernels) may import, call or link it, and it
imports nothing from that package.

Everything is plain NumPy in float64 (the compact-page format's own steps in
binary32, as the format defines them).  Parity of every function here is
pinned by the ``-m "not gpu"`` tests in ``tests/test_oracle_pins.py`` and
``tests/test_oracle_compact_pins.py`` (brute force, closed forms, invariants,
a published check value and library second opinions); no function is
"parity unpinned".
"""

from .paged_attention import (  # noqa: F401
    bf16_bits_to_f64,
    request_history,
    attention,
    tile_attention,
    lse_merge,
    decode_layer,
    merge_stress_partials,
    softmax_union,
)
from . import compact_pages  # noqa: F401,E402
