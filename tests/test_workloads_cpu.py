"""The algorithmic bytes and flops behind every roofline fraction the bench
reports, pinned to values worked out by hand for each workload (the workload
shapes: Llama-3-8B attention, 32/8 heads, D = 128, H = 4096; the fp16 MHA
shapes, 32/32 heads, D = 64, H = 2048; the tiny decode, 8/2 heads, D = 64,
H = 512).  The literals below are written out, not recomputed by the
formulas under test."""
import pytest

from zero_copy_offloaded_gb300 import workloads as wl

W = wl.WORKLOADS


def test_decode_host_bytes():
    # K and V prefix of every (sequence, KV head) read once; one row appended each
    assert W["tiny_decode"].host_read_bytes() == 1 << 20                 # 1 MiB
    assert W["tiny_decode"].host_write_bytes() == 512                    # 2 x 2 heads x 64 x 2 B
    assert W["llama8b_decode"].host_read_bytes() == 1 << 30              # 1 GiB
    assert W["llama8b_decode"].host_write_bytes() == 32 << 10            # 32 KiB
    assert W["mha_fp16_decode"].host_read_bytes() == 1 << 30             # 16 x 32 x 8192 x 64
    assert W["longctx_b4_s128k"].host_read_bytes() == 2 << 30            # B*S*4 KiB = 2 GiB
    assert W["longctx_b1_s16k"].host_read_bytes() == 64 << 20            # 64 MiB


def test_prefill_host_bytes():
    p = W["llama8b_prefill"]
    assert p.host_read_bytes() == 112 << 20    # 2 x 8 heads x 28672 x 128 x 2 B
    assert p.host_write_bytes() == 16 << 20    # 2 x 8 heads x 4096 x 128 x 2 B
    m = W["mha_fp16_prefill"]
    assert m.host_read_bytes() == 96 << 20     # 2 x 2 seq x 32 heads x 6144 x 64 x 2 B
    assert m.host_write_bytes() == 32 << 20


def test_prefill_flops():
    p = W["llama8b_prefill"]
    # causal (query, key) pairs per head: T*P + T(T+1)/2 = 4096*28672 + 4096*4097/2
    assert p.attn_pairs() == 125_831_168
    assert p.attn_flops() == 2_061_617_856_512          # x 32 heads x 4 x 128
    assert p.proj_flops() == 206_158_430_208            # 2 x 4096 x 4096 x (4096 + 2 x 1024)
    assert p.flops() == pytest.approx(2.268e12, rel=1e-3)
    m = W["mha_fp16_prefill"]
    assert m.attn_pairs() == 29_362_176                 # 2 x (2048*6144 + 2048*2049/2)
    assert m.attn_flops() == 240_534_945_792            # x 32 heads x 4 x 64
    assert m.proj_flops() == 103_079_215_104            # 2 x 4096 x 2048 x 96 x 64


def test_prefill_hbm_minimum():
    # x 32 MiB + weights 48 MiB + Q written and read 64 MiB + out 32 MiB
    assert W["llama8b_prefill"].hbm_min_bytes() == 176 << 20


def test_decode_attention_flops():
    # 4 x B x Hq x (P + 1) x D: the new token attends to itself
    assert W["llama8b_decode"].attn_flops() == 4 * 8 * 32 * 32769 * 128


def test_prefill_partial_rows_hand_worked():
    """Partial rows of the KV-stationary prefill (256-key chunks): the 112
    wholly cached chunks are seen by all 4096 tokens, new-token chunk i by
    4096 - 256 i of them; 32 query heads; 260 bytes per row (fp16 o + lse)."""
    import bench
    w = W["llama8b_prefill"]
    rows = (112 * 4096 + sum(4096 - 256 * i for i in range(16))) * 32
    assert rows == 15_794_176
    assert bench.prefill_partial_rows(w) == rows
    assert rows * 260 == 4_106_485_760   # the combine's reads (ncu: 4,106,566,144 B)
    q = W["llama8b_prefill_quarter"]
    assert bench.prefill_partial_rows(q) == (28 * 1024 + 1024 + 768 + 512 + 256) * 32
