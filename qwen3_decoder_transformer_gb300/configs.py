"""Model shapes and workloads used by the tests and the benchmark.

Shapes follow the Qwen3 config fields (hidden_size, num_hidden_layers, num_attention_heads,
num_key_value_heads, head_dim, intermediate_size, vocab_size, rope_theta, rms_norm_eps,
tie_word_embeddings) as listed in "A modern architecture: Qwen3" (the 0.6B contract) and the
model table of "Transformer architectures: modern" (Qwen3 0.6B and 8B rows).
"""
from __future__ import annotations

TINY = dict(name="tiny-2L-d256", n_layers=2, hidden=256, n_q_heads=8, n_kv_heads=4, head_dim=64,
            intermediate=768, vocab=1024, tie_embeddings=False, rope_theta=1e6, rms_eps=1e-6,
            max_positions=4096)

QWEN3_0P6B = dict(name="qwen3-0.6b-shape", n_layers=28, hidden=1024, n_q_heads=16, n_kv_heads=8,
                  head_dim=128, intermediate=3072, vocab=151936, tie_embeddings=True,
                  rope_theta=1e6, rms_eps=1e-6, max_positions=40960)

QWEN3_8B = dict(name="qwen3-8b-shape", n_layers=36, hidden=4096, n_q_heads=32, n_kv_heads=8,
                head_dim=128, intermediate=12288, vocab=151936, tie_embeddings=False,
                rope_theta=1e6, rms_eps=1e-6, max_positions=40960)

# Workloads: prefill batch x tokens, then optional decode at a pre-filled context.
WORKLOADS = {
    "tiny": dict(model=TINY, seed=0, prefill=(1, 64), decode_steps=8, decode_batch=1,
                 prefilled_ctx=0),
    "0.6b-prefill-1x2048": dict(model=QWEN3_0P6B, seed=1, prefill=(1, 2048), decode_steps=0,
                                decode_batch=0, prefilled_ctx=0),
    "0.6b-prefill-8x4096-decode-64@4096": dict(model=QWEN3_0P6B, seed=2, prefill=(8, 4096),
                                               decode_steps=128, decode_batch=64,
                                               prefilled_ctx=4096),
    "8b-prefill-1x8192": dict(model=QWEN3_8B, seed=3, prefill=(1, 8192), decode_steps=0,
                              decode_batch=0, prefilled_ctx=0),
    "8b-prefill-1x32768-decode-16@32768": dict(model=QWEN3_8B, seed=4, prefill=(1, 32768),
                                               decode_steps=64, decode_batch=16,
                                               prefilled_ctx=32768),
}
