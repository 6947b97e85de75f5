"""Host-side logic of the benchmark: the algorithmic byte counts behind every
roofline fraction, and the source hash that ties a recorded ncu traffic figure
to the kernels it was taken on.

The byte counts are checked against tensor-by-tensor lists written out here
(every input read once, every output written once, with element sizes bf16 2,
e4m3 1, e2m1 1/2, fp32 4, e4m3 scale factor 1), so that a dropped or doubled
tensor in the formulas shows up.
"""
import json
import os

import pytest

import bench

R, T, H = 8, 4096, 7168


def _nbytes(*tensors):
    total = 0
    for shape, size in tensors:
        n = 1
        for d in shape:
            n *= d
        total += n * size
    return int(total)


def test_headline_bytes():
    want = _nbytes(*[((T, H), 2)] * R,         # partials
                   ((T, H), 2), ((H,), 2),     # residual, gamma
                   ((T, H), 2), ((T, H), 2))   # residual_out, norm_out
    assert bench.fused_bytes(1, R, T, H) == want
    # with the optional allreduce_out as well
    assert bench.fused_bytes(1, R, T, H, allreduce_out=True) == want + T * H * 2


def test_allreduce_only_bytes():
    assert bench.fused_bytes(0, R, T, H) == _nbytes(*[((T, H), 2)] * R, ((T, H), 2))


@pytest.mark.parametrize("pattern", range(2, 9))
def test_quantising_pattern_bytes(pattern):
    P = 1024
    reads = [((T, H), 2)] * R + [((T, H), 2), ((H,), 2)]
    writes = [((T, H), 2)]  # residual_out
    if pattern in (2, 3, 4, 5):
        reads.append(((1,), 4))  # the global scale factor
    if pattern in (4, 5):
        writes.append(((T, H), 2))  # norm_out
    if pattern in (7, 8):
        writes.append(((T, P), 2))  # partial_norm_out
    if pattern in (2, 4):
        writes.append(((T, H), 1))
    if pattern in (6, 7):
        writes += [((T, H), 1), ((T, H // 128), 4)]
    if pattern in (3, 5):
        writes += [((T, H), 0.5), ((T, H // 16), 1)]  # LINEAR scale factors
    assert bench.fused_bytes(pattern, R, T, H, P=P) == _nbytes(*reads, *writes)


@pytest.mark.parametrize("layout,rows", [(0, 128), (1, 40)])
def test_swizzled_scale_factor_padding_is_counted(layout, rows):
    """T=37, H=320: 20 scale factors per row padded to 20 columns; rows padded
    to the 128- or 8-row tile."""
    t, h = 37, 320
    base = bench.fused_bytes(3, 2, t, h, sf_layout=2) - t * (h // 16)
    assert bench.fused_bytes(3, 2, t, h, sf_layout=layout) == base + rows * 20


def test_sharded_norm_bytes():
    Q, K = 1024, 128
    assert bench.qk_bytes(R, T, Q, K) == _nbytes(((T, R * (Q + K)), 2), ((T, R * (Q + K)), 2),
                                                 ((R * (Q + K),), 2))
    assert bench.rms_sharded_bytes(R, T, 768) == _nbytes(((T, R * 768), 2), ((T, R * 768), 2), ((R * 768,), 2))


def test_reduce_scatter_bytes_over_all_ranks():
    """R calls, one per rank's slice: each partial row read once, add_in and
    residual once, gamma once per call."""
    want = _nbytes(*[((T, H), 2)] * R, ((T, H), 2), ((T, H), 2), ((R, H), 2),
                   ((T, H), 2), ((T, H), 2))
    assert bench.rs_add_bytes(R, T, H) == want
    want8 = want - T * H * 2 + _nbytes(((T, H), 1), ((T, H // 128), 4))
    assert bench.rs_add_bytes(R, T, H, fp8_block=True) == want8


def test_allgather_bytes():
    t, q, kv, rope = 65536, 1536, 512, 64
    hid = q + kv + rope
    assert bench.ag_bytes(0, t, q, kv, rope) == _nbytes(((t, hid), 2), ((t, hid), 2))
    assert bench.ag_bytes(1, t, q, kv, rope) == _nbytes(((t, hid), 2), ((t, hid), 2), ((t, q), 2), ((t, kv), 2),
                                                        ((q,), 2), ((kv,), 2))
    assert bench.ag_bytes(2, t, q, kv, rope) == _nbytes(((t, hid), 2), ((t, hid), 2), ((t, kv), 2), ((t, q), 1),
                                                        ((t, q // 128), 4), ((q,), 2), ((kv,), 2))


def test_roofline_entry_arithmetic():
    e = bench.roofline_entry(7_000_000_000, 1.0, 7000.0)
    assert e["gbs"] == pytest.approx(7000.0) and e["frac"] == pytest.approx(1.0) and e["us"] == 1000.0


def test_code_tokens_ignore_comments_and_layout():
    a = "int f(int x) {\n  // doubles x\n  return 2 * x; /* ok */\n}\n"
    b = "int f(int x)\n{\n    /* twice x,\n       as before */ return 2 * x;\n}"
    assert bench._code_tokens(a) == bench._code_tokens(b)
    assert bench._code_tokens(a) != bench._code_tokens(a.replace("2 * x", "3 * x"))


def test_code_tokens_keep_literals():
    src = 'asm("ld.global.cs.v4.u32 {%0}, [%1]; // not a comment"); char c = \'"\'; // gone'
    out = bench._code_tokens(src)
    assert "// not a comment" in out and "gone" not in out and "'\"'" in out


def test_recorded_traffic_table_is_well_formed():
    """Every record names a benchmark row, a positive byte count, the 16-digit
    hash of its kernel family's sources and a committed profile summary."""
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    rows = bench._case_builders()
    for key, row in rec["rows"].items():
        assert key in rows, key
        assert isinstance(row["bytes"], int) and row["bytes"] > 0, key
        assert len(row["kernel_hash"]) == 16 and int(row["kernel_hash"], 16) >= 0
        assert os.path.exists(os.path.join(bench.ROOT, "profiles", row["profile"])), row["profile"]


def test_kernel_families_cover_the_sources():
    fams = set()
    for files in bench.KERNEL_FAMILIES.values():
        fams.update(files)
    assert fams == set(bench.KERNEL_SOURCES)
    assert bench.row_family("ag-rms-fp8b") == "ag_norm" and bench.row_family("c5-qk") == "qk_norm"
    assert bench.row_family("c3-p7") == "fused_rows" and bench.row_family("rs-add") == "fused_rows"


def test_sweep_shapes_are_valid_calls():
    """Every (pattern, R, H) of ``--sweep-t`` is a call the library accepts:
    H a multiple of the pattern's quantisation group, R and H in range."""
    group = {3: 16, 5: 16, 6: 128, 7: 128}
    for p, R, H in bench.SWEEP_SHAPES:
        assert 0 <= p <= 8 and 1 <= R <= 16 and 8 <= H <= 16384
        assert H % group.get(p, 8) == 0, (p, H)
    assert list(bench.SWEEP_TOKENS) == sorted(set(bench.SWEEP_TOKENS)) and bench.SWEEP_TOKENS[0] >= 1


def test_gpus_flag_is_honoured():
    """--gpus N: one process runs as is; N > 1 outside torchrun starts N ranks;
    under torchrun N must equal WORLD_SIZE, else the bench exits with an error."""
    assert bench.check_world(1, {}) == "run"
    assert bench.check_world(4, {}) == "spawn"
    assert bench.check_world(2, {"WORLD_SIZE": "2"}) == "run"
    assert bench.check_world(1, {"WORLD_SIZE": "1"}) == "run"
    for gpus, world in ((2, "4"), (1, "2"), (8, "1")):
        with pytest.raises(SystemExit):
            bench.check_world(gpus, {"WORLD_SIZE": world})
    with pytest.raises(SystemExit):
        bench.check_world(0, {})


def test_spawn_command_starts_n_local_ranks():
    cmd = bench.spawn_command(["--gpus", "4", "--steps", "7"], 4, 29512)
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node=4" in cmd and "--nnodes=1" in cmd
    assert "--master-addr=127.0.0.1" in cmd and "--master-port=29512" in cmd
    assert cmd[-4:] == ["--gpus", "4", "--steps", "7"] and cmd[-5].endswith("bench.py")


def test_headline_is_the_largest_workload_and_both_arms_share_its_config():
    """The headline step is pattern 7 on R=8 T=8192 H=7168: the largest
    per-call byte count among the patterns that workload is measured on (FP8
    per tensor, FP8 1x128, PartialOut with and without FP8 1x128), and the
    reference arm prints the same config as ours."""
    from reduce_residual_rmsnorm_gb300 import workloads as wl

    c3 = wl.WORKLOADS["C3"]
    assert bench.headline_bytes() == bench.fused_bytes(7, c3.R, c3.T, c3.H, 1024) == 1251751936
    for p in (2, 6, 8):
        assert bench.fused_bytes(p, c3.R, c3.T, c3.H, 1024) < bench.headline_bytes()
    c2 = wl.WORKLOADS["C2"]
    assert bench.fused_bytes(1, c2.R, c2.T, c2.H) < bench.headline_bytes()
    cfg = bench.headline_config(1)
    assert (cfg["pattern"], cfg["R"], cfg["T"], cfg["H"], cfg["partial_cols"]) == (7, 8, 8192, 7168, 1024)
    assert cfg["bytes_per_step"] == bench.headline_bytes() and cfg == bench.headline_config(1)


def test_every_bench_row_names_a_builder():
    rows = bench._case_builders()
    assert "c3-p7" in rows and "c2-p1" in rows
    for key, (label, build) in rows.items():
        assert label and callable(build)
