"""Host logic of bench.py that needs no GPU: workload naming and the lookup
of committed ncu summaries."""
import os
import types

import bench
from synth import gen


def _args(q6_scales):
    return types.SimpleNamespace(q6_scales=q6_scales)


def test_workload_name_marks_int8_scales_on_q6k_only():
    q6 = gen.config_by_name("q6_K_ffn_down_3584x18944_nt2630")
    q4 = gen.config_by_name("q4_K_qproj_3584x3584_nt512")
    assert bench._workload_name(q6, _args("small")) == q6.name
    assert bench._workload_name(q6, _args("int8")) == q6.name + "_int8scales"
    assert bench._workload_name(q4, _args("int8")) == q4.name


def test_profile_lookup_is_by_exact_kernel_and_workload():
    # a summary exists for the fp16-plane kernel on the q-proj workload; none
    # for another kernel on it, and none for a made-up workload
    assert bench._profiled_traffic("q4_K_qproj_3584x3584_nt512", "no_such_kernel") is None
    assert bench._profiled_traffic("no_such_workload", "mmq_gemm_kernel") is None
    p = os.path.join(bench.ROOT, "profiles", "mmq_gemm_kernel_q4_K_qproj_3584x3584_nt512.md")
    assert os.path.exists(p)
    got = bench._profiled_traffic("q4_K_qproj_3584x3584_nt512", "mmq_gemm_kernel")
    # a number when the summary was taken on the current source, else None
    text = open(p).read()
    current = bench._code_sha1(os.path.join(bench.ROOT, "quantized_int8_gemm_gb300", "csrc", "gemm.cu"))
    assert (got is not None) == (current in text)
    if got is not None:
        assert got > 0


def test_code_hash_ignores_comments(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    a.write_text('int f() { return 1; }  // one\n/* block */ const char *s = "//x";\n')
    b.write_text('int f() {   return 1; }\n const char *s = "//x";  // other comment\n')
    assert bench._code_sha1(str(a)) == bench._code_sha1(str(b))
    b.write_text('int f() { return 2; }\n const char *s = "//x";\n')
    assert bench._code_sha1(str(a)) != bench._code_sha1(str(b))


def test_nt_override_renames_the_workload(monkeypatch):
    """--nt keeps the workload's shape and generators and renames its _nt suffix."""
    got = {}
    monkeypatch.setattr(bench, "run_reference", lambda args, cfg, rank: got.setdefault("cfg", cfg))
    bench.main(["--impl", "reference", "--workload", "q6_K_qproj_3584x3584_nt512", "--nt", "16"])
    cfg = got["cfg"]
    assert (cfg.name, cfg.nt, cfg.od, cfg.id, cfg.qtype) == ("q6_K_qproj_3584x3584_nt16", 16, 3584, 3584, "q6_K")


def test_arm_option_sets_the_flags_every_call_passes(monkeypatch):
    """--arm forces one GEMM arm for the run (the C ABI's MMQ_ARM_* values)."""
    monkeypatch.setattr(bench, "run_reference", lambda args, cfg, rank: None)
    try:
        for name, flag in (("pair", 4), ("split", 3), ("f16", 1), ("auto", 0)):
            bench.main(["--impl", "reference", "--arm", name])
            assert bench.ARM[0] == flag
    finally:
        bench.ARM[0] = 0
