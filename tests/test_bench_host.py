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
    # one launch, captured with no cross-kernel prefetch, reads the gate/up weights
    # once (234.9 MB) and the activations, and writes the SwiGLU activations
    assert 234_881_024 <= traffic <= 234_881_024 * 1.03
    assert "profiles/gemm_swapab_llama8b_m5.md" in src


def test_both_arms_describe_the_same_workload(monkeypatch, capsys):
    """The reference arm's line carries the GPU arm's config object, so the driver
    compares the same workload, and it times every layer (no projection from a
    sample): the sampler is built with all of the model's layers."""
    import json
    import sys

    seen = {}

    class FakeSample:
        def __init__(self, args):
            seen["layers"] = args.cpu_layers

        def step(self):
            return 0.5, 3, 0.5

        def describe(self):
            return "stand-in"

    monkeypatch.setattr(bench, "OracleSample", FakeSample)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "4", "--warmup", "1"])
    args = bench.parse_args()
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    bench.run_reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert seen["layers"] == args.layers == 32
    assert line["config"] == bench.workload_config(args, 1)
    assert line["impl"] == "reference" and line["ms_per_step"] == 500.0 and line["value"] == 6.0
