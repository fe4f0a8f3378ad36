"""The bench's byte model against the byte figures the pages print.

* radiance_lmhead_int4.py, module docstring: the 248320 x 5120 head in int4
  with group-128 bf16 scales moves 656 MB per call; per-channel fp8 moves
  1.27 GB; against bf16 the int4 head frees 1.88 "GiB" (the figure is GB --
  a garbled unit) and 0.61 against fp8.
* "Fused WNA16 GEMM for tied quantized lm_head logits", reviewer comment
  items 1-2: the 151936 x 2048 fp16 logits GEMV moves 622 MB; its int8 copy
  is a 311 MB weight; rescoring the top 8 reads 32 KB.
"""
import bench


def test_int4_head_bytes_per_call():
    b = bench.logits_bytes(1, 248320, 5120, 4, 128, out_bytes=2, x_bytes=2, scale_bytes=2)
    assert b == 656_071_680
    assert round(b / 1e6) == 656


def test_weight_sizes_and_savings():
    n, k = 248320, 5120
    int4 = n * k // 2 + n * (k // 128) * 2          # codes + bf16 scales
    fp8 = n * k
    bf16 = n * k * 2
    assert round(fp8 / 1e9, 2) == 1.27
    # the docstring's "1.88 GiB" and "0.61 GiB" are these GB figures cut to two
    # decimals (in GiB they would read 1.76 and 0.57)
    assert int((bf16 - int4) / 1e7) / 100 == 1.88
    assert int((fp8 - int4) / 1e7) / 100 == 0.61
    assert round((bf16 - int4) / 2**30, 2) == 1.76


def test_int8_head_and_rescore_bytes():
    n, k = 151936, 2048
    assert round(n * k * 2 / 1e6) == 622                       # the fp16 GEMV's weight
    w8 = bench.logits_bytes(1, n, k, 8, 0, scale_bytes=2) - (k * 2 + n * 2 + n * 2)
    assert w8 == n * k and round(w8 / 1e6) == 311              # int8 codes
    assert bench.rescore_bytes(1, k, 8) - (k * 2 + 8 * 10) == 32_768   # 8 rows of 2048 fp16
