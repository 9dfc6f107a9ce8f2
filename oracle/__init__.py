"""fp64 CPU oracle for bf16 forward attention.

TEST INFRASTRUCTURE. This package exists to check the CUDA path. Only the tests,
the smoke check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may
import it. The product (``bf16_forward_attention_gb300``) never imports it, and it
imports nothing from the product: the two share no code. The only thing both sides
use is the seeded input generator, which holds none of the method's arithmetic.

What it computes is the plain definition O = softmax(Q K^T * scale) V, in fp64,
then rounded once to bf16 per mode. Sources: the snilld.dk article "Open source
attention-kernel i HIP slaar AITER v3 paa MI300X" (sections "Hvad er udgivet",
"Hvordan kernen arbejder", "Numerik samlet eet sted") and the tilnote.io note on
MoonMath AI's HIP attention kernel for MI300X (section on the performance figures
and the kernel's scope).
"""
from .attention import (  # noqa: F401
    MODES,
    attention_fp64,
    attention_rows_fp64,
    attention_varlen_fp64,
    bf16_bits_to_f64,
    nonfinite_bits,
    round_bf16,
    to_bhsd,
    ulp_distance,
)
