"""Host-side pieces of the bench (no GPU): the identity of the projection code an
ncu capture came from, and the traffic lookup that depends on it."""
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_code_sha1_ignores_comments_and_blank_lines(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    c = tmp_path / "c.cu"
    a.write_text("int f(int x) {\n  return x + 1;  // one more\n}\n")
    b.write_text("// header comment\n\nint f(int x) {\n\n  return x + 1;  // a different remark\n}\n")
    c.write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert bench.code_sha1(str(a)) == bench.code_sha1(str(b))
    assert bench.code_sha1(str(a)) != bench.code_sha1(str(c))


def test_committed_gemm_profile_matches_the_code():
    """The committed ncu summary of the projection kernel was captured from the code
    as it stands, so the bench reports its traffic (a stale one would read null)."""
    traffic, src = bench.profiled_traffic("gate_up")
    assert traffic is not None, src
    # one launch reads the gate/up weights once (234.9 MB) plus the 16 MB L2 prefetch
    # of the next projection, and writes the activations
    assert 234_881_024 <= traffic <= 234_881_024 + 16_000_000 + 8_000_000
    assert "profiles/gemm_swapab_llama8b_m5.md" in src
