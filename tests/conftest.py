import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """Error reports of the session's GEMM parity checks: the gated count
    (fail, against the unrounded FP64 reference) and the count measured against
    the reference rounded to BF16 (fail_literal_bf16_ref, reported only)."""
    gu = sys.modules.get("tests.gpu_util")
    reps = getattr(gu, "REPORTS", None) if gu else None
    if not reps:
        return
    tr = terminalreporter
    tr.write_sep("-", "GEMM parity reports (entries checked / fail / fail against BF16(ref))")
    tot = [0, 0, 0]
    for what, r in reps:
        tot[0] += r["n"]
        tot[1] += r["fail"]
        tot[2] += r["fail_literal_bf16_ref"]
        tr.write_line(f"{what}: n={r['n']} fail={r['fail']} fail_literal_bf16_ref={r['fail_literal_bf16_ref']} "
                      f"max_abs={r['max_abs']:.3g} nrmse={r['nrmse']:.3g}")
    tr.write_line(f"total: {len(reps)} checks, n={tot[0]} fail={tot[1]} fail_literal_bf16_ref={tot[2]}")
