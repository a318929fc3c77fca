"""Host-side logic of the benchmark (no GPU): the per-row DRAM traffic attribution that feeds the
roofline's `traffic` figure."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_write_traffic_rows(tmp_path, monkeypatch):
    bench = load_bench()
    out = tmp_path / "traffic.txt"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(out))
    hdr = '"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"\n'
    lines = [hdr]

    def launch(i, name, mb_read, mb_write):
        lines.append('"%d","%s","gpu__time_duration.sum","us","10"\n' % (i, name))
        lines.append('"%d","%s","dram__bytes_read.sum","Mbyte","%s"\n' % (i, name, mb_read))
        lines.append('"%d","%s","dram__bytes_write.sum","Mbyte","%s"\n' % (i, name, mb_write))

    n = 0
    for step in range(2):                                   # two steps
        launch(n, "void k_index_block_scores<64, 2, 32>(const CUtensorMap_st)", 80, 8); n += 1
        for _ in range(4):
            launch(n, "k_attn_plan(const int *, long)", 1, 0); n += 1
            launch(n, "void k_attn_kvouter<128>(CUtensorMap_st)", 1000, 1000); n += 1
        launch(n, "void k_decode_tail<128, 0>(AttnParams)", 2, 0); n += 1
    for _ in range(3):                                      # three loss calls, two gradient calls
        launch(n, "void k_kl_kvouter<128, 8, 0>(KlQMaps)", 19000, 200); n += 1
    for _ in range(2):
        launch(n, "void k_kl_kvouter<128, 8, 1>(KlQMaps)", 20000, 2000); n += 1
        launch(n, "k_kl_dq_merge(const int *)", 2000, 100); n += 1
    csv = tmp_path / "t.csv"
    csv.write_text("".join(lines))
    bench.write_traffic(str(csv), "test command")
    rows = {l.split()[0]: int(l.split()[1]) for l in out.read_text().splitlines()
            if l and not l.startswith("#")}
    assert rows["index_branch"] == 88_000_000
    assert rows["main_branch"] == 4 * (1_000_000 + 2_000_000_000)
    assert rows["decode"] == 2_000_000
    assert rows["kl_loss_fwd"] == 19_200_000_000              # per loss call (3 calls)
    assert rows["kl_loss_bwd"] == 22_000_000_000 + 2_100_000_000   # gradient pass + dQ merge
    # a capture of a smaller case scaled by 4 updates only the rows asked for
    bench.write_traffic(str(csv), "smaller case", scale=4.0, only={"main_branch"}, tag="B")
    text = out.read_text()
    rows2 = {l.split()[0]: l.split() for l in text.splitlines() if l and not l.startswith("#")}
    assert int(rows2["main_branch"][1]) == 4 * rows["main_branch"] and rows2["main_branch"][3] == "B"
    assert int(rows2["decode"][1]) == rows["decode"] and rows2["decode"][3] == "A"
    assert "# capture A: test command" in text and "# capture B: smaller case" in text


def test_roofline_row_peaks():
    """Tensor-bound rows divide by the burst bf16 figure and give the sustained fraction beside
    it; HBM-bound rows divide by the measured copy bandwidth."""
    bench = load_bench()
    pk = dict(hbm=6000.0, bf16=2000.0, bf16_sust=1600.0, src="measured")
    t = bench.roofline_row("main_branch", 2.0, "tensor", 2.0e12, "TFLOP/s", pk)
    assert t["achieved"] == 1000.0 and t["peak"] == 2000.0 and t["frac"] == 0.5
    assert t["frac_of_sustained"] == 0.625 and "burst" in t["peak_source"]
    h = bench.roofline_row("decode", 0.1, "hbm", 3.0e8, "GB/s", pk)
    assert h["achieved"] == 3000.0 and h["frac"] == 0.5 and "frac_of_sustained" not in h


def test_write_traffic_adds_per_kernel_captures(tmp_path, monkeypatch):
    """One capture per kernel of the same step add up to the step's figure; ncu's own messages
    and the program's output in an ncu stdout CSV are skipped; a capture label that no row uses
    any more is dropped from the notes."""
    bench = load_bench()
    out = tmp_path / "traffic.txt"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(out))
    hdr = '"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"\n'

    def capture(path, name, mb_read, mb_write):
        path.write_text(
            '{"metric": "program output on stdout"}\n==PROF== Connected to process 1\n' + hdr +
            '"0","%s","gpu__time_duration.sum","us","10"\n' % name +
            '"0","%s","dram__bytes_read.sum","Mbyte","%s"\n' % (name, mb_read) +
            '"0","%s","dram__bytes_write.sum","Mbyte","%s"\n' % (name, mb_write))

    paths = []
    for n, (name, r, w) in enumerate([("void k_index_block_scores<64, 1, 24>(CUtensorMap_st)", 20, 1),
                                      ("void k_attn_kvouter<128, 8>(CUtensorMap_st)", 900, 1500),
                                      ("void k_attn_shared<128>(CUtensorMap_st)", 2000, 300),
                                      ("k_attn_plan(const int *, long)", 10, 5)]):
        p = tmp_path / ("c%d.csv" % n)
        capture(p, name, r, w)
        paths.append(str(p))
    bench.write_traffic(",".join(paths), "per-kernel captures", scale=4.0, tag="C")
    rows = {l.split()[0]: l.split() for l in out.read_text().splitlines()
            if l and not l.startswith("#")}
    assert int(rows["index_branch"][1]) == 4 * 21_000_000
    assert int(rows["main_branch"][1]) == 4 * (2_400_000_000 + 2_300_000_000 + 15_000_000)
    # a second capture of the same rows under another label replaces the first label's note
    bench.write_traffic(",".join(paths), "again", scale=4.0, tag="E")
    text = out.read_text()
    assert "# capture E: again" in text and "# capture C:" not in text
