"""The benchmark's own bookkeeping, on the CPU: the algorithmic byte model of
a step and the parsing of the clock samples taken during the timed region."""

import pytest

import bench


@pytest.mark.parametrize("pattern, calls, step", [
    ([False, False, False, False], [6, 10, 10, 10], 30),   # norm fused into the stored last pass
    ([False, False, False, True], [6, 10, 10, 6], 32),     # last micro-batch deferred (the bench's default)
    ([True, True, True, True], [0, 0, 0, 8], 34),          # every gradient resident
    ([True], [2], 28),                                      # one micro-batch, deferred
    ([True, False, True, True], [0, 8, 0, 8], 34),          # pairs
    ([True] * 7 + [False] + [True] * 8, [0] * 7 + [20] + [0] * 7 + [20], 46),
])
def test_pass_bytes(pattern, calls, step):
    """Stored pass: acc (if it holds earlier micro-batches) + 2 B per folded
    gradient read, 4 B written; deferred LAST: the same reads, no write; step:
    acc?, the pending gradients and p, m, v read (12 B), p, m, v, bf16 written
    (14 B)."""
    got_calls, got_step = bench.pass_bytes(pattern)
    assert got_calls == calls and got_step == step


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def _clocks_from(rows):
    c = bench.Clocks(0, enabled=True)
    c.f.write("\n".join(rows) + "\n")
    c.p = _Done()
    return c.stop()


ROW = "0, {sm}, 2070, {pw}, 0x0, {hw}, Not Active, Not Active, {cap}"


def test_clocks_median_under_load_and_reasons():
    rows = [ROW.format(sm=2070, pw=900.0, hw="Not Active", cap="Not Active")] * 5 + \
           [ROW.format(sm=1500, pw=120.0, hw="Not Active", cap="Not Active")] * 3 + \
           [ROW.format(sm=1900, pw=1390.0, hw="Active", cap="Active")]
    r = _clocks_from(rows)
    assert r["sm_mhz"] == 2070 and r["sm_max_mhz"] == 2070
    assert r["samples"] == 9 and r["samples_under_load"] == 6      # idle samples (<= 300 W) left out
    assert r["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert r["power_w_max"] == 1390.0


def test_clocks_no_reasons():
    r = _clocks_from([ROW.format(sm=2070, pw=850.0, hw="Not Active", cap="Not Active")] * 4)
    assert r["reasons"] == [] and r["samples_under_load"] == 4


def test_kernel_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    """The recorded-profile hash follows the kernels' code, not their comments."""
    f = tmp_path / "k.cuh"
    monkeypatch.setattr(bench, "KERNEL_SOURCES", [str(f)])
    f.write_text("// header\n__global__ void k(float *p) { p[0] = 1.0f; }  /* body */\n")
    h0 = bench.kernel_hash()
    f.write_text("// another header\n/* reworded\n   block */ __global__ void k(float *p) {\n  p[0] = 1.0f;\n}\n")
    assert bench.kernel_hash() == h0
    f.write_text("__global__ void k(float *p) { p[0] = 2.0f; }\n")
    assert bench.kernel_hash() != h0
