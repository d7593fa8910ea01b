"""The algorithmic byte counts behind the bench's roofline fractions, pinned to
figures worked out by hand from the layouts (B = 1 sequence, Hk = 16, Hv = 32,
dk = dv = 128, bf16 activations, fp32 outputs; Mamba2: 8 groups, 128 heads,
N = 128, P = 64)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_decode_bytes_per_token():
    # state 2 * 32 * 128 * 128 * s, q and k 2 * 16 * 128 * 2, v 32 * 128 * 2, a and b 2 * 32 * 2,
    # output 32 * 128 * 4, slot 4
    assert bench.decode_bytes_per_token(4) == 4_194_304 + 8_192 + 8_192 + 128 + 16_384 + 4 == 4_227_204
    assert bench.decode_bytes_per_token(2) == 2_097_152 + 8_192 + 8_192 + 128 + 16_384 + 4 == 2_130_052


def test_replay_unit_bytes():
    # per (sequence, value head): S0 128 * 128 * s; an entry is a raw key (256) and an fp32 record
    # {alpha, beta, 1/|k|, 0, w[128]} (528); a token's inputs are its share of q and k (2 * 256 / 2),
    # v (256), a and b (4); an appended entry is raw k, raw v and a record (1,040); the output 512;
    # the two pointers 16
    token = 256 + 256 + 4
    assert bench.replay_unit_bytes(7, 1, False, 4) == 65_536 + 7 * 784 + token + 1_040 + 512 + 16 == 73_108
    assert bench.replay_unit_bytes(16, 1, True, 4) == 2 * 65_536 + 16 * 784 + token + 1_040 + 512 + 16
    assert bench.replay_unit_bytes(3, 4, False, 2) == 32_768 + 3 * 784 + 4 * (token + 1_040 + 512) + 16
    # a bf16 read copy over an fp32 master: the copy read when not folding; on a fold the master read
    # and written and the copy written
    assert bench.replay_unit_bytes(7, 1, False, 4, read_bytes=2) == 32_768 + 7 * 784 + token + 1_040 + 512 + 16
    assert bench.replay_unit_bytes(16, 1, True, 4, read_bytes=2) == (16_384 * 10 + 16 * 784 + token + 1_040 +
                                                                     512 + 16)


def test_spec_bytes_per_window():
    # the source state read and T = 4 copies written (32 * 128 * 128 * s each), T tokens of inputs
    # (16,512 each), T outputs (16,384 each), T + 1 slot indices
    assert bench.spec_bytes_per_seq(4, 4) == 5 * 2_097_152 + 4 * 16_512 + 4 * 16_384 + 20 == 10_617_364
    assert bench.spec_bytes_per_seq(4, 2) == 5 * 1_048_576 + 4 * 16_512 + 4 * 16_384 + 20 == 5_374_484


def test_mamba2_bytes():
    # decode: state 2 * 128 * 128 * 64 * s, B and C 2 * 8 * 128 * 2, x 128 * 64 * 2, dt 128 * 2,
    # output 128 * 64 * 4, slot 4
    assert bench.mamba2_decode_bytes_per_token(4) == 8_388_608 + 4_096 + 16_384 + 256 + 32_768 + 4 == 8_442_116
    # replay, per (sequence, head): S0 128 * 64 * s; an entry is raw B (256) and a record
    # {alpha, delta, 1, 0, w[64]} (272); the token's share of B and C (2 * 256 / 16), x (128), dt (2);
    # the appended entry raw B, raw x and a record (656); the output 256; the pointers 16
    assert bench.mamba2_replay_unit_bytes(7, False, 4) == 32_768 + 7 * 528 + 32 + 128 + 2 + 656 + 256 + 16
    assert bench.mamba2_replay_unit_bytes(16, True, 2) == 2 * 16_384 + 16 * 528 + 162 + 656 + 256 + 16


def test_prefill_counts():
    # MMA flops of the tensor-core prefill, per chunk of 64 tokens and 128 state rows:
    # 2 * (128*128*128 + 128*64*128 + 2 * 128*64*64 + 128*128*64) = 2 * 5,242,880 = 10,485,760;
    # 19 sequences x 32 heads x 32 chunks of the 2048-token workload
    assert bench.prefill_mma_flops(1, 1, 128, 64) == 10_485_760
    assert bench.prefill_mma_flops(19, 32, 128, 2048) == 19 * 32 * 32 * 10_485_760 == 204_010_946_560
    # a ragged last chunk counts as a chunk; dv = 256 is two row blocks; an interval of 16 makes chunks of 16
    assert bench.prefill_mma_flops(1, 1, 128, 65) == 2 * 10_485_760
    assert bench.prefill_mma_flops(1, 1, 256, 64) == 2 * 10_485_760
    assert bench.prefill_mma_flops(1, 1, 128, 64, interval=16) == 4 * 10_485_760
    # HBM bytes: per token q and k (2 * 16 * 128 * 2), v (32 * 128 * 2), a and b (2 * 32 * 2), the fp32
    # output (32 * 128 * 4); per (sequence, head) the state read and written (2 * 128 * 128 * s)
    per_token = 8_192 + 8_192 + 128 + 16_384
    assert bench.prefill_bytes(1, 16, 32, 128, 128, 1, 4) == per_token + 2 * 32 * 65_536
    assert bench.prefill_bytes(19, 16, 32, 128, 128, 2048, 2) == 19 * 2048 * per_token + 2 * 19 * 32 * 32_768
