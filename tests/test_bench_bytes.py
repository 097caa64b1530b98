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
