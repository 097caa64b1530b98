"""The benchmark's algorithmic byte counts and hop roles (CPU only): the
roofline fractions it prints divide these bytes by measured launch times,
so they are checked here against the message layout and the schedules."""
import bench
import oracle


def test_ring_roles_and_dar_bytes():
    roles = bench.hop_roles(False, 16)
    assert roles[0] == ("compress", False, 1.0)
    assert roles[1:] == [("dar", False, 1.0)] * 15
    m = 177.0                                  # message bytes per super-group at 5 bits
    # message in + bf16 gradient + mean and perm + message out
    assert bench.launch_bytes(1, 10, m) == 10 * (m + 512 + 8 + m)
    assert bench.launch_bytes(0, 10, m) == 10 * (512 + m + 8)


def test_butterfly_roles_follow_the_schedule():
    # N = 8: compress of the sent half, step 1 (bf16 addend, split), step 2
    # (fp32 addend, split), step 3 (the owner's single quantization)
    assert [r[0] for r in bench.hop_roles(True, 8)] == ["compress", "dar_bf16_split", "dar_f32_split",
                                                         "dar_f32_final"]
    assert [r[0] for r in bench.hop_roles(True, 2)] == ["compress", "dar_bf16_final"]
    m = 177.0
    # split step with fp32 addend: message in, fp32 partial + perm, half sent, half kept as fp32
    got = bench.launch_bytes(1, 8, m, fp32_addend=True, send_frac=0.5)
    assert got == 8 * (m + 1024 + 4) + 4 * m + 4 * 1024


def test_message_bytes_per_super_group_at_five_bits():
    # all-4-bit and all-8-bit mixes that average 5 bits: 0.691 B per coordinate
    n4, n8 = 3 * 1024, 1024
    per = oracle.message_bytes(0, n4, n8) / (n4 + n8) / 256
    assert abs(per - (5 + 17 * 8 / 256) / 8) < 1e-3


def test_pipelined_launches_count_the_fused_round_bytes():
    # the logged super-groups of a pipelined round add up to J (N + 1), and
    # the bytes are the fused ring's for the same round
    J, N, m = 1000, 16, 177.0
    assert bench.launch_bytes(8, J * (N + 1), m, n_ranks=N) == bench.launch_bytes(7, J * (N + 1), m, n_ranks=N)
    parts = [J * (N + 1) // 5] * 4
    parts.append(J * (N + 1) - sum(parts))
    total = sum(bench.launch_bytes(8, p, m, n_ranks=N) for p in parts)
    assert abs(total - bench.launch_bytes(8, J * (N + 1), m, n_ranks=N)) < 1e-6 * total


def test_exchange_mode_picks_by_size():
    from quantized_hop_gradient_gb300.allreduce import FUSED_MAX_SG, exchange_mode, pipeline_parts
    assert exchange_mode(8, True, 1 << 20) == (False, None)          # butterfly: step by step
    assert exchange_mode(65, False, 1 << 20) == (False, None)        # beyond 64 ranks
    assert exchange_mode(8, False, FUSED_MAX_SG) == (True, None)
    assert exchange_mode(16, False, 3905805) == (False, 32)          # Gemma-1B ring of 16: 2N parts
    assert exchange_mode(8, False, 1309148) == (False, 11)           # BERT-large ring of 8: about N sqrt(units) / 144
    assert FUSED_MAX_SG == 1 << 16
    assert pipeline_parts(8, FUSED_MAX_SG + 1) == 1                  # one part up to 16,384 units
    assert pipeline_parts(16, 32 * 16384) == 1 and pipeline_parts(16, 32 * 16385) == 14
    assert pipeline_parts(8, 1 << 20) == 10 and pipeline_parts(16, 1 << 21) == 28
    assert pipeline_parts(64, 1 << 26) == 128
    assert pipeline_parts(4, 1) == 1
