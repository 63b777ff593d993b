"""CPU oracle for the KV4-RL decode hot path — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (``libkv4`` and the
``int8_hybrid_paged_gb300`` binding) never does.
"""
from .kv4_oracle import (  # noqa: F401
    PV_FLOAT,
    PV_INTEGER,
    RD,
    RN,
    RU,
    OracleCache,
    bf16_to_f32,
    exp2f,
    f16_bits_to_f64,
    f32_to_bf16_rn,
    f32_to_f16,
    fwht128,
    load,
    num_threads,
    quant_affine,
    quant_query,
    rope128,
    e4m3_rn,
    e4m3_value,
    e2m1_rn,
    e2m1_value,
    quant_nvfp4,
    quant_mxfp4,
)
