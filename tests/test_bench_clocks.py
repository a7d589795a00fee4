"""The bench's clock record: medians of the samples taken inside the timed
window, throttle reasons seen, and the memory clock and power beside the
SM clock (CPU only; the samples are synthetic nvidia-smi rows)."""
import bench

ROW = "0, {sm}, 2032, {w}, 0x4, Not Active, Not Active, Not Active, {cap}, {mem}"


def _sampler(rows, times):
    c = bench.ClockSampler(0)
    c.samples = [(t, [p.strip() for p in r.split(",")]) for t, r in zip(times, rows)]
    return c


def test_summary_medians_reasons_and_window():
    rows = [ROW.format(sm=1600, w=1050.0, cap="Active", mem=3996),
            ROW.format(sm=1580, w=1040.0, cap="Active", mem=3996),
            ROW.format(sm=1620, w=1060.0, cap="Not Active", mem=3996),
            ROW.format(sm=300, w=90.0, cap="Not Active", mem=405)]  # idle, long after the window
    c = _sampler(rows, [10.0, 10.05, 10.1, 20.0])
    c.mark(10.0, 10.1)
    s = c.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 1600 and s["sm_max_mhz"] == 2032
    assert s["mem_mhz"] == 3996 and s["power_w"] == 1050.0
    assert s["reasons"] == ["sw_power_cap"]


def test_rows_without_memory_clock_still_summarise():
    rows = [r.rsplit(",", 1)[0] for r in (ROW.format(sm=1590, w=1000.0, cap="Active", mem=0),) * 2]
    c = _sampler(rows, [5.0, 5.05])
    c.mark(5.0, 5.05)
    s = c.summary()
    assert s["sm_mhz"] == 1590 and s["mem_mhz"] is None and s["reasons"] == ["sw_power_cap"]


def test_no_samples_reads_unsampled():
    c = _sampler([], [])
    c.mark(0.0, 1.0)
    assert c.summary()["reasons"] == ["unsampled"]
