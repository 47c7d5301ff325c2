"""CPU oracle for paged-KV attention (TEST INFRASTRUCTURE).

Only ``tests/``, the smoke check in ``__graft_entry__`` and the CPU-baseline
leg of ``bench.py`` may import this package.  The product path never does,
and this package imports nothing from the product.
"""
from .paged_attention import (  # noqa: F401
    gather_request_kv, visible_keys, softmax_attention, paged_attention,
    paged_decode, visible_block_range, splitk_partials, lse_combine,
    run_batch,
)
from .brute_force import brute_force_attention  # noqa: F401
from .kv_append import kv_append  # noqa: F401
from .key_mass import key_mass  # noqa: F401
from .rope_norm import rms_norm, rope, kv_append_rope  # noqa: F401
