"""Summaries of Nsight Compute output for the FLCE kernels.

  python -m linear_cross_entropy_token_gb300.ncu_summary launches <launches.csv>
      per kernel kind: launches, total device time, share (from an
      `ncu --metrics gpu__time_duration.sum --csv --log-file` launch list)
  python -m linear_cross_entropy_token_gb300.ncu_summary raw <report.ncu-rep>
      per captured launch: duration, DRAM bytes, tensor-pipe and memory
      utilisation, warp stalls (from `ncu -i <rep> --page raw --csv
      --print-units base`)
  python -m linear_cross_entropy_token_gb300.ncu_summary traffic <report.ncu-rep>
        [--workload NAME --chunk C --chunks K --dlogits MODE]
      DRAM bytes per launch per kernel kind, as JSON (K: chunks of the call
      whose first launches were captured; weights dW's store against its adds)
"""
from __future__ import annotations

import collections
import csv
import io
import json
import re
import subprocess
import sys

_GEMM = {(0, 0, 0): "gemm_logits_lse", (0, 0, 3): "gemm_dlogits_recompute", (0, 1, 2): "gemm_dx",
         (0, 1, 1): "gemm_dx_bf16", (1, 1, 2): "gemm_dw", (0, 0, 2): "gemm_check_kk",
         (1, 0, 2): "gemm_check_mk"}
_PLAIN = {"combine_dlogits_bf16_kernel": "combine_dlogits",   # before its substring below
          "count_valid_kernel": "count_valid", "lse_combine_kernel": "lse_combine",
          "dlogits_bf16_kernel": "dlogits_inplace", "dlogits_f32_kernel": "dlogits_inplace_f32",
          "dx_reduce_kernel": "dx_split_reduce", "loss_finalize_kernel": "loss_finalize",
          "simt_gemm_f32_kernel": "simt_gemm_f32", "simt_tile_stats_kernel": "simt_tile_stats_f32",
          "simt_splitk_reduce_kernel": "simt_splitk_reduce_f32",
          "wait_check_kernel": "wait_check", "umma_pair_dual_kernel": "gemm_dx_dw",
          "umma_wide_dual_kernel": "gemm_dx_dw",
          "device_result_kernel": "device_result"}

RAW_METRICS = [
    ("gpu__time_duration.sum", "time_us", 1e-3),
    ("dram__bytes_read.sum", "dram_read_MB", 1e-6),
    ("dram__bytes_write.sum", "dram_write_MB", 1e-6),
    ("gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed", "dram_%", 1.0),
    ("sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active", "tensor_pipe_%", 1.0),
    ("sm__throughput.avg.pct_of_peak_sustained_elapsed", "sm_throughput_%", 1.0),
    ("l1tex__data_bank_conflicts_pipe_lsu_mem_shared.sum", "smem_bank_conflicts", 1.0),
    ("launch__registers_per_thread", "regs", 1.0),
    ("sm__cycles_elapsed.avg.per_second", "sm_GHz", 1e-9),
]


def kind_of(name: str) -> str:
    m = re.search(r"umma_(?:gemm|pair|wide)_kernel<(\d+), (\d+), (\d+)>", name)
    if m:
        return _GEMM.get(tuple(int(v) for v in m.groups()), "gemm_other")
    for k, v in _PLAIN.items():
        if k in name:
            return v
    return name.split("(")[0][-60:]


def launches(csv_path: str):
    hdr = None
    agg = collections.OrderedDict()
    with open(csv_path) as f:
        for r in csv.reader(f):
            if r and r[0] == "ID":
                hdr = r
                continue
            if not hdr or len(r) != len(hdr):
                continue
            d = dict(zip(hdr, r))
            if d.get("Metric Name") != "gpu__time_duration.sum":
                continue
            scale = {"ns": 1.0, "us": 1e3, "usecond": 1e3, "ms": 1e6, "msecond": 1e6}.get(
                d.get("Metric Unit", "ns"), 1.0)
            a = agg.setdefault(kind_of(d["Kernel Name"]), [0, 0.0])
            a[0] += 1
            a[1] += float(d["Metric Value"].replace(",", "")) * scale
    total = sum(v[1] for v in agg.values()) or 1.0
    return [(k, n, t, t / total) for k, (n, t) in agg.items()]


def raw(rep_path: str):
    out = subprocess.run(["ncu", "-i", rep_path, "--page", "raw", "--csv", "--print-units", "base"],
                         capture_output=True, text=True, check=True).stdout
    rows = list(csv.reader(io.StringIO(out)))
    hdr = rows[0]
    res = []
    for r in rows[2:]:
        d = {"kernel": kind_of(r[hdr.index("Kernel Name")])}
        for metric, label, scale in RAW_METRICS:
            if metric in hdr:
                v = r[hdr.index(metric)].replace(",", "")
                try:
                    d[label] = float(v) * scale
                except ValueError:
                    d[label] = None
        stalls = {h.split("stalled_")[1].split("_per_issue")[0]: r[i]
                  for i, h in enumerate(hdr)
                  if h.startswith("smsp__average_warps_issue_stalled_") and h.endswith("_per_issue_active.ratio")}
        top = sorted(((float(v), k) for k, v in stalls.items() if v not in ("", "n/a")), reverse=True)[:4]
        d["top_stalls"] = ", ".join(f"{k} {v:.2f}" for v, k in top)
        res.append(d)
    return res


def traffic(rep_path: str, chunks: int = 0):
    """DRAM bytes per launch per kernel kind. With chunks = K > 0 the capture
    holds the first chunks of one call: the dW GEMM's first launch stores dW
    and its later ones add into it, so its per-launch figure is the mean over
    a K-chunk call, (first + (K - 1) x mean of the others) / K; the same for
    the launch that runs the dx and dW GEMMs together."""
    per = collections.OrderedDict()
    for d in raw(rep_path):
        if d.get("dram_read_MB") is None:
            continue
        per.setdefault(d["kernel"], []).append((d["dram_read_MB"] + d["dram_write_MB"]) * 1e6)
    out = {}
    for k, v in per.items():
        if chunks > 0 and k in ("gemm_dw", "gemm_dx_dw") and len(v) > 1:
            per_launch = (v[0] + (chunks - 1) * sum(v[1:]) / len(v[1:])) / chunks
        else:
            per_launch = sum(v) / len(v)
        out[k] = {"launches": len(v), "dram_bytes_per_launch": per_launch}
    return out


def _md_table(header, rows) -> str:
    lines = ["| " + " | ".join(header) + " |", "|" + "---|" * len(header)]
    lines += ["| " + " | ".join(str(c) for c in r) + " |" for r in rows]
    return "\n".join(lines)


def main(argv=None):
    argv = argv or sys.argv[1:]
    if not argv:
        print(__doc__)
        return 2
    cmd, path = argv[0], argv[1]
    if cmd == "launches":
        rows = [(k, n, f"{t / 1e6:.3f}", f"{100 * s:.2f}%") for k, n, t, s in launches(path)]
        print(_md_table(["kernel", "launches", "total ms", "share"], rows))
    elif cmd == "raw":
        res = raw(path)
        keys = ["kernel"] + [lab for _, lab, _ in RAW_METRICS if any(lab in d for d in res)] + ["top_stalls"]
        fmt = lambda v: f"{v:.4g}" if isinstance(v, float) else str(v)
        print(_md_table(keys, [[fmt(d.get(k)) for k in keys] for d in res]))
    elif cmd == "traffic":
        # optional: --workload NAME --chunk C, recorded with the kernel source hash
        opts = dict(zip(argv[2::2], argv[3::2]))
        from .build import source_hash
        out = {"workload": opts.get("--workload"), "chunk": int(opts.get("--chunk", 0)),
               "dlogits": opts.get("--dlogits", "inplace"),
               "source_hash": source_hash(),
               "kernels": traffic(path, int(opts.get("--chunks", 0)))}
        print(json.dumps(out, indent=1))
    else:
        print(__doc__)
        return 2
    return 0


if __name__ == "__main__":
    sys.exit(main())
