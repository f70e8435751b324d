"""The C-ABI boundary on the CPU: libc3.so loads without a GPU, exports every
entry point include/c3_api.h declares, the ctypes records match the C layout
(checked by compiling a probe against the header with gcc), and argument
errors come back as the documented status codes before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "c3_api.h")


@pytest.fixture(scope="module")
def c3():
    from concurrent_communication_overlap_gb300 import build
    build.build()
    from concurrent_communication_overlap_gb300 import c3 as mod
    return mod


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(c3_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(c3):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(c3.lib(), n), n
    assert set(names) == set(c3.EXPORTED)


def test_record_layouts_match_the_header(c3, tmp_path):
    probe = tmp_path / "probe.c"
    probe.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "c3_api.h"
#define F(T, f) printf(#T "." #f " %zu\n", offsetof(T, f))
int main(void) {
  printf("c3_problem %zu\nc3_timing %zu\nc3_device_info %zu\n", sizeof(c3_problem), sizeof(c3_timing), sizeof(c3_device_info));
  F(c3_problem, coll); F(c3_problem, shards); F(c3_problem, unit_bytes); F(c3_problem, nranks);
  F(c3_problem, sm_kernel); F(c3_problem, flush_buf); F(c3_problem, stream);
  F(c3_problem, settle_us); F(c3_problem, peak_flops); F(c3_problem, coll_plateau_ce);
  F(c3_problem, ce_stage); F(c3_problem, ce_stage_bytes);
  F(c3_timing, t_comm_ev); F(c3_timing, cls); F(c3_timing, smid_overlap); F(c3_timing, status);
  F(c3_timing, gemm_bound); F(c3_timing, coll_bound);
  F(c3_device_info, comm_default_sms);
  return 0;
}
''')
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), str(probe), "-o", str(exe)], check=True)
    got = dict(line.rsplit(" ", 1) for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                               check=True).stdout.split("\n") if line)
    assert int(got["c3_problem"]) == ctypes.sizeof(c3.C3Problem)
    assert int(got["c3_timing"]) == ctypes.sizeof(c3.C3Timing)
    assert int(got["c3_device_info"]) == ctypes.sizeof(c3.C3DeviceInfo)
    for key, val in got.items():
        if "." in key:
            rec, field = key.split(".")
            cls = {"c3_problem": c3.C3Problem, "c3_timing": c3.C3Timing, "c3_device_info": c3.C3DeviceInfo}[rec]
            assert getattr(cls, field).offset == int(val), key


def test_strerror_covers_every_status(c3):
    for code in (0, -1, -2, -3, -4, -5):
        assert c3.c3_strerror(code) not in ("", "unknown status")
    assert c3.c3_strerror(-99) == "unknown status"


def test_argument_errors_before_any_cuda_call(c3):
    # Each of these is rejected by host-side checks that run before the
    # library touches the device, so they are safe without a GPU.
    assert c3.c3_gemm(0x1000, 0x1000, 0x1000, -1, 4, 8, check=False) == c3.C3_EINVAL
    assert c3.c3_gemm(0x1000, 0x1000, 0x1000, 4, 4, 12, check=False) == c3.C3_EALIGN   # K % 8
    assert c3.c3_gemm(0x1008, 0x1000, 0x1000, 4, 4, 16, check=False) == c3.C3_EALIGN   # A misaligned
    assert c3.c3_gemm(0x1000, 0x1000, 0x1004, 4, 4, 16, check=False) == c3.C3_EALIGN   # C misaligned
    assert c3.c3_gemm(None, 0x1000, 0x1000, 4, 4, 16, check=False) == c3.C3_EINVAL
    assert c3.c3_gemm(0x1000, 0x1000, 0x1000, 4, 4, 16, sm_budget=-2, check=False) == c3.C3_EINVAL
    assert c3.c3_gemm(0x1000, 0x1000, 0x1000, 1 << 31, 4, 16, check=False) == c3.C3_EUNSUP
    assert c3.c3_gemm(None, None, None, 0, 5, 16, check=False) == c3.C3_OK   # empty: nothing to do
    shards = [0x10000 * (r + 1) for r in range(8)]
    assert c3.c3_allgather(shards, 0x100000, 24, 8, check=False) == c3.C3_EALIGN
    assert c3.c3_allgather(shards, 0x100008, 32, 8, check=False) == c3.C3_EALIGN
    assert c3.c3_allgather(shards[:1] + [0x10008] + shards[2:], 0x100000, 32, 8, check=False) == c3.C3_EALIGN
    assert c3.c3_allgather(shards[:1] + [None] + shards[2:], 0x100000, 32, 8, check=False) == c3.C3_EINVAL
    assert c3.c3_allgather(shards, 0x100000, 32, 0, check=False) == c3.C3_EINVAL
    assert c3.c3_allgather(shards, 0x10000, 32, 8, check=False) == c3.C3_EINVAL        # out overlaps shard 0
    assert c3.c3_allgather(shards, 0x100000, 32, 8, engine=7, check=False) == c3.C3_EINVAL
    assert c3.c3_allgather(shards, 0x100000, 0, 8, check=False) == c3.C3_OK            # empty collective
    assert c3.c3_alltoall(0x10000, 0x20000, 32, 9, check=False) == c3.C3_EINVAL        # 81 blocks > 64
    assert c3.c3_alltoall(0x10000, 0x10400, 32, 8, check=False) == c3.C3_EINVAL        # in/out overlap
    assert c3.c3_alltoall(0x10000, 0x20000, 40, 8, check=False) == c3.C3_EALIGN
    assert c3.c3_alltoall(0x10000, 0x20000, 0, 8, check=False) == c3.C3_OK
    ins = [0x10000 * (r + 1) for r in range(8)]
    assert c3.c3_allreduce(ins, 0x200000, 33, 8, check=False) == c3.C3_EALIGN        # count % 32
    assert c3.c3_allreduce(ins, 0x200000, 64, 9, check=False) == c3.C3_EINVAL        # > 8 ranks
    assert c3.c3_allreduce(ins, 0x10000, 64, 8, check=False) == c3.C3_EINVAL         # out overlaps input 0
    assert c3.c3_allreduce(ins[:1] + [0x20004] + ins[2:], 0x200000, 64, 8, check=False) == c3.C3_EALIGN
    assert c3.c3_allreduce(ins, 0x200000, 0, 8, check=False) == c3.C3_OK
    assert c3.c3_gemm_noalloc(0x1000, 0x1000, 0x1000, -1, 4, 8, check=False) == c3.C3_EINVAL
    assert c3.c3_gemm_noalloc(0x1000, 0x1000, 0x1000, 4, 4, 12, check=False) == c3.C3_EALIGN
    assert c3.c3_gemm_noalloc(None, None, None, 4, 0, 8, check=False) == c3.C3_OK
    assert c3.c3_selftest_wait(0, 0) == c3.C3_EINVAL
    assert c3.c3_selftest_wait(6_000_000_000, 0) == c3.C3_EINVAL
    assert c3.c3_selftest_wait(1000, 2) == c3.C3_EINVAL
    assert c3.lib().c3_l2_flush(0x1001, 64, None) == c3.C3_EALIGN
    assert c3.lib().c3_l2_flush(None, 64, None) == c3.C3_EINVAL
    assert c3.lib().c3_inject_fault(5) == c3.C3_EINVAL
    assert c3.lib().c3_inject_fault(-1) == c3.C3_EINVAL
    assert c3.lib().c3_inject_fault(c3.C3_FAULT_GEMM_LAUNCH) == c3.C3_OK
    assert c3.lib().c3_inject_fault(c3.C3_FAULT_NONE) == c3.C3_OK   # disarmed again
    n = ctypes.c_int()
    arr = (c3.C3CtaWindow * 4)()
    assert c3.lib().c3_cta_windows(2, arr, 4, ctypes.byref(n)) == c3.C3_EINVAL
    assert c3.lib().c3_cta_windows(0, None, 4, ctypes.byref(n)) == c3.C3_EINVAL
    assert c3.lib().c3_cta_windows(0, arr, -1, ctypes.byref(n)) == c3.C3_EINVAL


def test_run_and_time_reject_bad_records(c3):
    p = c3.Problem(0x1000, 0x2000, 0x3000, 4, 4, 16, c3.C3_COLL_ALLGATHER, 0x100000, 32,
                   shards=[0x10000 * (r + 1) for r in range(8)])
    t = c3.C3Timing()
    assert c3.lib().c3_run(ctypes.byref(p.rec), 9, 0, 0, ctypes.byref(t)) == c3.C3_EINVAL
    assert c3.lib().c3_run(ctypes.byref(p.rec), 1, 0, 2, ctypes.byref(t)) == c3.C3_EINVAL
    assert c3.lib().c3_run(None, 1, 0, 0, ctypes.byref(t)) == c3.C3_EINVAL
    arr = (c3.C3Timing * 1)()
    assert c3.lib().c3_time(ctypes.byref(p.rec), 1, 0, 0, 0, 0, arr) == c3.C3_EINVAL
    bad = c3.Problem(0x1000, 0x2000, 0x3000, 4, 4, 16, 5, 0x100000, 32, shards=[0x10000] * 8)
    assert c3.lib().c3_run(ctypes.byref(bad.rec), 1, 0, 0, ctypes.byref(t)) == c3.C3_EINVAL
    overlap = c3.Problem(0x1000, 0x2000, 0x100000, 4, 4, 16, c3.C3_COLL_ALLGATHER, 0x100000, 32,
                         shards=[0x10000 * (r + 1) for r in range(8)])
    assert c3.lib().c3_run(ctypes.byref(overlap.rec), 1, 0, 0, ctypes.byref(t)) == c3.C3_EINVAL
    # timer options: settle period and the rates of the taxonomy's bounds
    for kw in ({"settle_us": -1}, {"settle_us": 1000001}, {"peak_flops": -1.0}, {"peak_bytes_per_s": float("nan")},
               {"coll_plateau_sm": float("inf")}, {"coll_plateau_ce": -2.0}):
        q = c3.Problem(0x1000, 0x2000, 0x3000, 4, 4, 16, c3.C3_COLL_ALLGATHER, 0x100000, 32,
                       shards=[0x10000 * (r + 1) for r in range(8)], **kw)
        assert c3.lib().c3_time(ctypes.byref(q.rec), 1, 0, 0, 0, 1, arr) == c3.C3_EINVAL, kw
        assert c3.lib().c3_run(ctypes.byref(q.rec), 1, 0, 0, ctypes.byref(t)) == c3.C3_EINVAL, kw
    # the host-staged copy-engine variant needs a 16-byte aligned bounce buffer of the copies' size
    # (8 shards x 32 bytes here); an unknown variant is rejected
    for kw, want in (({"ce_variant": 5}, c3.C3_EINVAL),
                     ({"ce_variant": c3.C3_CE_HOST_STAGED}, c3.C3_EINVAL),
                     ({"ce_variant": c3.C3_CE_HOST_STAGED, "ce_stage": (0x200000, 8 * 32 - 16)}, c3.C3_EINVAL),
                     ({"ce_variant": c3.C3_CE_HOST_STAGED, "ce_stage": (0x200008, 8 * 32)}, c3.C3_EALIGN)):
        q = c3.Problem(0x1000, 0x2000, 0x3000, 4, 4, 16, c3.C3_COLL_ALLGATHER, 0x100000, 32,
                       shards=[0x10000 * (r + 1) for r in range(8)], **kw)
        assert c3.lib().c3_run(ctypes.byref(q.rec), 2, 0, 0, ctypes.byref(t)) == want, kw
        assert c3.lib().c3_time(ctypes.byref(q.rec), 2, 0, 0, 0, 1, arr) == want, kw


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    import importlib.util
    src = os.path.join(ROOT, "concurrent_communication_overlap_gb300", "c3.py")
    dst = tmp_path / "c3_copy.py"
    dst.write_text(open(src).read())
    spec = importlib.util.spec_from_file_location("c3_copy", dst)
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)
