"""Host-side arithmetic of bench.py (CPU only): the per-step byte and flop counts and the launch
counts that go into the JSON line."""

import bench
from weight_linear_attention_gb300 import inputs as I


def test_launches_per_call():
    W = I.WORKLOADS
    assert bench._launches_per_call(W["f1_b8h12t1024_bf16"], 6) == 1          # fused kernel
    # scan path, Falcon-3 at 8192 tokens per call, chunk 32: normalisers, tensor-core maps, the CUDA-core
    # map kernel (strong-decay chunks only), compose, groups, apply
    assert bench._launches_per_call(W["f3w4_b2h12t16384_bf16"], 5) == 6
    assert bench._launches_per_call(W["f3aw4_b2h12t16384_bf16"], 5) == 5     # no normaliser pass
    assert bench._launches_per_call(W["f3w4_b2h12t16384_bf16"].with_(seqlen=256), 5) == 4  # one group
    assert bench._launches_per_call(W["f3w4_b2h12t16384_bf16"].with_(chunk=16), 5) == 5  # CUDA-core maps only


def test_forward_algorithmic_bytes():
    w = I.WORKLOADS["f1_b8h12t1024_bf16"]
    tok = 8 * 12 * 1024
    # q, k, v and out in bf16, beta and lambda fp32, S_final fp32, the tail key
    expect = tok * (3 * 64 + 64) * 2 + tok * 8 + 96 * 64 * 64 * 4 + 96 * 64 * 2
    assert bench._algorithmic_bytes(w, 2) == expect
    # Falcon-2 and 2A read beta per value column
    for name in ("f2_b8h12t2048_bf16", "f2a_b8h12t2048_bf16"):
        w2 = I.WORKLOADS[name]
        tok2 = 8 * 12 * 2048
        assert bench._algorithmic_bytes(w2, 2) == tok2 * (3 * 64 + 64) * 2 + tok2 * (64 + 1) * 4 + \
            96 * 64 * 64 * 4 + 96 * 64 * 2


def test_backward_counts():
    w = I.WORKLOADS["f1_bwd_b8h12t1024_bf16"]
    one = 2 * 64 ** 3
    assert bench._bwd_flops_per_chunk(w) == one * (10 + 1 / 3 + 2 + 15)
    assert bench._bwd_flops_per_chunk(I.WORKLOADS["f1a_bwd_b8h12t1024_bf16"]) == one * 13
    tok = 8 * 12 * 1024
    # q, k, v, dout (bf16) and beta, lambda read; fp32 dq, dk, dv, dbeta, dlambda written; dS_final, dS0
    expect = tok * 4 * 64 * 2 + tok * 8 + tok * 3 * 64 * 4 + tok * 8 + 2 * 96 * 64 * 64 * 4
    assert bench._bwd_bytes(w, 2) == expect
    # a call runs its sequences in groups on streams of their own, three kernels each
    assert [bench._bwd_groups(n) for n in (1, 3, 4, 15, 16, 96)] == [1, 1, 2, 2, 4, 4]


def test_chunk_flops():
    # Falcon-1 at the 130M shape: per chunk-head 2 (4 C^2 d + 2 C d^2 + C^2 d / 2) with C = d = 64
    w = I.WORKLOADS["f1_b8h12t1024_bf16"]
    per = 2 * (4 * 64 ** 3 + 2 * 64 ** 3 + 64 ** 3 / 2)
    assert bench._chunk_flops(w) == per * 96 * 16
    assert abs(bench._chunk_flops(w) - 5.2e9) < 0.1e9  # ~5.2 GFLOP of chunk algebra for this config
    assert bench._chunk_flops(I.WORKLOADS["f1a_b8h12t1024_bf16"]) == 2 * 4 * 64 ** 3 * 96 * 16
    # Falcon-2 / 2A: the same products at their own length
    assert bench._chunk_flops(I.WORKLOADS["f2_b8h12t2048_bf16"]) == per * 96 * 32
    assert bench._chunk_flops(I.WORKLOADS["f2a_b8h12t2048_bf16"]) == 2 * 4 * 64 ** 3 * 96 * 32
    # Falcon-3 at W = 4, C = 32: R = 128 windowed rows per chunk, 24 sequences x 512 chunks
    R, C, d = 128, 32, 64
    per3 = 2 * (1.5 * R * R * d + 2 * C * R * d + 2 * R * d * d + C * d * d)
    assert bench._chunk_flops(I.WORKLOADS["f3w4_b2h12t16384_bf16"]) == per3 * 24 * 512
    assert abs(bench._chunk_flops(I.WORKLOADS["f3w4_b2h12t16384_bf16"]) - 80.5e9) < 0.1e9
    assert bench._chunk_flops(I.WORKLOADS["f3aw4_b2h12t16384_bf16"]) == 2 * (2 * C * R * d + C * d * d + R * d * d) * 24 * 512
