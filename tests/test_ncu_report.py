"""The ncu summary writer (mla_verify_attention_gb300.ncu_report) on small,
hand-written CSV files in the layout ncu --csv --log-file produces: per-kernel
launch counts, totals and shares, the split kernel's DRAM bytes and
tensor-pipe activity, and the source hash that bench.py checks before it
reports the recorded traffic."""
import json
import os

from mla_verify_attention_gb300 import ncu_report

HEADER = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
          '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
          '"Metric Value"\n')


def _row(i, kernel, metric, unit, value):
    return ('"%d","1","python3","127.0.0.1","%s","1","7","(384, 1, 1)","(150, 1, 1)","0","10.3",'
            '"Command line profiler metrics","%s","%s","%s"\n' % (i, kernel, metric, unit, value))


SPLIT = "void mla::verify_split_kernel<0, true>(CUtensorMap_st, CUtensorMap_st, mla::SplitParams)"
MERGE = "void mla::combine_kernel<16, 1>(mla::CombineParams)"


def test_summary_from_csv(tmp_path):
    src = tmp_path / "raw"
    src.mkdir()
    with open(src / "launches_chain9_p256.csv", "w") as fh:
        fh.write("==PROF== Connected to process 1\n" + HEADER)
        for i in range(3):
            fh.write(_row(2 * i, SPLIT, "gpu__time_duration.sum", "us", "10.0"))
            fh.write(_row(2 * i + 1, MERGE, "gpu__time_duration.sum", "ns", "2,500"))
    with open(src / "counters_chain9_p256.csv", "w") as fh:
        fh.write(HEADER)
        for i in range(2):
            fh.write(_row(i, SPLIT, "dram__bytes_read.sum", "Mbyte", "0.5"))
            fh.write(_row(i, SPLIT, "dram__bytes_write.sum", "byte", "1000"))
            fh.write(_row(i, SPLIT, "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active",
                          "%", "40"))
    prof = tmp_path / "profiles"
    t = ncu_report.summarize("chain9_p256", str(src), str(prof))
    ll = t["launch_list"]
    assert ll["verify_split_kernel<0, true>"]["launches"] == 3
    assert abs(ll["verify_split_kernel<0, true>"]["total_us"] - 30.0) < 1e-9
    assert abs(ll["combine_kernel<16, 1>"]["avg_us"] - 2.5) < 1e-9      # ns and thousands separator
    assert abs(ll["verify_split_kernel<0, true>"]["share"] - 0.8) < 1e-9
    s = t["verify_split_kernel"]
    assert s["captured_launches"] == 2 and s["dram_bytes_per_launch"] == 501000.0
    assert s["tensor_pipe_active_pct"] == 40.0
    # 265 keys x 1152 bytes, read once
    assert t["algorithmic"]["cache_bytes_per_launch"] == 265 * 1152
    on_disk = json.load(open(prof / "traffic_chain9_p256.json"))
    assert on_disk["verify_split_kernel"]["dram_bytes_per_launch"] == 501000.0
    md = open(prof / "verify_call_chain9_p256_launches.md").read()
    assert "verify_split_kernel<0, true>" in md and "80.0 %" in md
    assert os.path.basename(str(prof / "traffic_chain9_p256.json")) in os.listdir(prof)


def test_short_kernel_names():
    assert ncu_report.short_name(SPLIT) == "verify_split_kernel<0, true>"
    assert ncu_report.short_name("void verify_split_kernel<0, 0>(CUtensorMap_st, SplitParams)") == \
        "verify_split_kernel<0, 0>"
    assert ncu_report.short_name("plain_kernel(int)") == "plain_kernel"
