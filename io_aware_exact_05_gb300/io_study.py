"""IO study of the attention backward: memory traffic of the tiled (fused)
backward against the materialise-P backward, over sequence length n and
head dim d.

"On the fine-grained I/O complexity of attention backward passes"
(Theorem 1.1) bounds the backward's IO with a cache of M words by
Theta(min{(n^2 d^2 + n d^3) / M, (n^2 d + n d^2) / sqrt(M)}), the first term
for M = Omega(d^2), where tiling as FlashAttention does is optimal; the
materialise-P backward (the small-cache algorithm's explicit n x n
matrices) moves Theta(n^2) words through memory whatever M is.

Two levels are measured, per kernel launch, with the GPU's counters:
  * DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum), and
  * L2 <-> SM bytes (lts__t_bytes.sum: every byte the SMs read from or write
    to L2), the traffic between the SMs' on-chip memory (shared memory and
    tensor memory, the "cache" of the theorem) and the memory beneath it.

Run one path and configuration per process under ncu, then summarise:

    ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,lts__t_bytes.sum \\
        --clock-control none --csv --log-file io_fused_n4096_d128.csv \\
        python -m io_aware_exact_05_gb300.io_study run --path fused --n 4096 --d 128
    (same with --path mat into io_mat_n4096_d128.csv)
    python -m io_aware_exact_05_gb300.io_study summarize io_*.csv

`run` does one forward and one backward of the path on B=1, H=4 synthetic
heads, non-causal (--B, --H, --causal change that).  `summarize` sums the backward launches of each file
(fused: every launch after the forward kernel; materialise-P: every launch
after its three forward launches) and prints bytes per path with reference
counts: the compulsory bytes and n^2 d^2 / M with M the K, V tile a CTA keeps
on chip.

Tile-size axis (the theorem's M at fixed n and d): `run --key-rows R` runs
the fused backward with key tiles of R = 128, 64 or 32 keys
(attn_bwd_dkdv_keys: a CTA keeps R keys' K and V rows on chip and streams
every Q and dO tile past them), captured on the key-tile kernel alone:

    ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,lts__t_bytes.sum \
        --clock-control none -k regex:bwd_kv --csv --log-file io_keys_n4096_d128_r64.csv \
        python -m io_aware_exact_05_gb300.io_study run --path fused --n 4096 --d 128 --key-rows 64
    python -m io_aware_exact_05_gb300.io_study keyrows io_keys_*.csv

`keyrows` prints, per (n, d, R), the kernel's bytes against n^2 d^2 / M with
M = 2 R d (the K and V rows the CTA keeps).

Sparse attention ("On the fine-grained I/O complexity of attention backward
passes", Theorem 4.5: Omega(min{Z_in^2 / M, Z_in sqrt(Z_QK) / sqrt(M)}) with
Z_in nonzero input entries and Z_QK kept score entries, split at
M = Z_in^2 / Z_QK): `run --path sparse --pattern W,G,R` runs the
block-sparse forward and backward over make_block_mask(n, W, G, R) (seed
3000 + n); capture the key-tile kernel and summarise with `sparse`, which
recomputes Z_QK from the same pattern and takes Z_in = n d (the inputs are
dense; with Z_QK = n^2 both terms become Theorem 1.1's).

`time --path fused|mat` times warm forward and backward calls of one path
with CUDA events (no profiler), for the fused vs materialise-P comparison.

`kernels` reads a launch list taken with
`ncu --metrics gpu__time_duration.sum,dram__bytes_read.sum,dram__bytes_write.sum`
and prints, per launch, its time, DRAM bytes and DRAM GB/s against the
measured HBM copy bandwidth (the bound of the HBM-bound kernels: the D
preprocess, the dQ conversion and the materialise-P row kernels).
"""

import argparse
import csv
import json
import os
import re
import sys

__all__ = ["main"]

B, H = 1, 4


def sparse_pattern(n, pattern):
    """The block pattern of a sparse IO-study run (uint8 [nb][nb])."""
    from .inputs import make_block_mask

    w_, g_, r_ = pattern
    return make_block_mask(n, w_, g_, r_, 3000 + n)


def _run(path, n, d, b=B, h=H, causal=False, dtype="bf16", key_rows=0, pattern=None):
    import torch

    from . import attn
    from .inputs import Workload, make_inputs

    w = Workload("io", b, h, n, d, dtype, causal, 1.0, 2000 + n + d)
    x = make_inputs(w)
    dev = torch.device("cuda", 0)
    q, k, v, do = (x[t].to(dev) for t in ("q", "k", "v", "do"))
    if path == "sparse":   # block-sparse forward and backward
        bm = sparse_pattern(n, pattern).to(dev)
        o, lse = attn.forward(q, k, v, causal=causal, block_mask=bm)
        attn.backward(q, k, v, o, do, lse, causal=causal, block_mask=bm)
    elif path == "fused" and key_rows:   # the backward's stages with R-key tiles
        o, lse = attn.forward(q, k, v, causal=causal)
        mode = attn.ATTN_DQ_PASS if d == 256 else attn.ATTN_DQ_ATOMIC
        ws = torch.empty(attn.attn_bwd_workspace_size(b, h, n, d, attn.ATTN_BF16, causal, mode),
                         dtype=torch.uint8, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        attn.attn_bwd_preprocess(o, do, lse, causal, mode, ws)
        attn.attn_bwd_dkdv_keys(q, k, v, do, dk, dv, w.scale, causal, mode, key_rows, ws)
        attn.attn_bwd_dq(q, k, v, do, dq, w.scale, causal, mode, ws)
    elif path == "fused":   # tiled forward, then the tiled backward (key-tile kernel + dQ)
        o, lse = attn.forward(q, k, v, causal=causal)
        attn.backward(q, k, v, o, do, lse, causal=causal)
    else:                 # materialise-P: S, P, dP, dS as n x n matrices in HBM
        ws = torch.empty(attn.attn_mat_workspace_size(b, h, n, d), dtype=torch.uint8,
                         device=dev)
        o, lse = torch.empty_like(q), torch.empty(b, h, n, device=dev)
        attn.attn_mat_fwd(q, k, v, o, lse, w.scale, causal, ws)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        attn.attn_mat_bwd(q, k, v, o, do, lse, dq, dk, dv, w.scale, causal, ws)
    torch.cuda.synchronize()
    rc = attn.attn_status()
    if rc:
        raise SystemExit("device status %d" % rc)


def _time(path, n, d, b, h, causal, reps=10):
    """Mean ms of the forward and of the backward of one path, warm, CUDA events."""
    import torch

    from . import attn
    from .inputs import Workload, make_inputs

    w = Workload("io", b, h, n, d, "bf16", causal, 1.0, 2000 + n + d)
    x = make_inputs(w)
    dev = torch.device("cuda", 0)
    q, k, v, do = (x[t].to(dev) for t in ("q", "k", "v", "do"))
    o, lse = torch.empty_like(q), torch.empty(b, h, n, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if path == "mat":
        ws = torch.empty(attn.attn_mat_workspace_size(b, h, n, d), dtype=torch.uint8, device=dev)
        fwd = lambda: attn.attn_mat_fwd(q, k, v, o, lse, w.scale, causal, ws)   # noqa: E731
        bwd = lambda: attn.attn_mat_bwd(q, k, v, o, do, lse, dq, dk, dv, w.scale, causal, ws)  # noqa: E731
    else:
        mode = attn.ATTN_DQ_AUTO
        ws = torch.empty(attn.attn_bwd_workspace_size(b, h, n, d, attn.ATTN_BF16, causal, mode),
                         dtype=torch.uint8, device=dev)
        fwd = lambda: attn.attn_fwd(q, k, v, o, lse, w.scale, causal)   # noqa: E731
        bwd = lambda: attn.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, w.scale, causal, mode, ws)  # noqa: E731
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for _ in range(3):
        fwd()
        bwd()
    torch.cuda.synchronize()
    tf = tb = 0.0
    for _ in range(reps):
        ev[0].record()
        fwd()
        ev[1].record()
        bwd()
        ev[2].record()
        torch.cuda.synchronize()
        tf += ev[0].elapsed_time(ev[1])
        tb += ev[1].elapsed_time(ev[2])
    if attn.attn_status():
        raise SystemExit("device status error")
    fl = 4 * b * h * n * n * d // (2 if causal else 1)
    out = {"path": path, "B": b, "H": h, "n": n, "d": d, "causal": causal,
           "fwd_ms": tf / reps, "bwd_ms": tb / reps,
           "fwd_tflops": fl / (tf / reps * 1e-3) / 1e12,
           "bwd_tflops": 2.5 * fl / (tb / reps * 1e-3) / 1e12}
    print(json.dumps(out))


def _rows(path):
    rows = list(csv.reader(open(path)))
    hi = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    h = rows[hi]
    ki, mi, ui, vi = (h.index("Kernel Name"), h.index("Metric Name"), h.index("Metric Unit"),
                      h.index("Metric Value"))
    idi = h.index("ID")
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9,   # bytes
             "ns": 1, "nsecond": 1, "us": 1e3, "usecond": 1e3, "ms": 1e6, "msecond": 1e6}   # ns
    launches = {}
    for r in rows[hi + 1:]:
        if len(r) <= vi:
            continue
        key = int(r[idi])
        name = r[ki].split("(")[0].split("<")[0].split("::")[-1].split()[-1]
        ent = launches.setdefault(key, {"name": name})
        ent[r[mi]] = float(r[vi].replace(",", "")) * scale.get(r[ui], 1)
    return [launches[k] for k in sorted(launches)]


def _bwd_bytes(path):
    """(DRAM bytes, L2 <-> SM bytes) summed over the backward launches."""
    ls = _rows(path)
    if "_fused_" in path:   # forward = fwd_tc_kernel, then the backward kernels
        first = next(i for i, l in enumerate(ls) if l["name"] == "fwd_tc_kernel") + 1
    else:                   # forward = S GEMM, row softmax, PV GEMM
        first = 3
    bwd = ls[first:]
    dram = sum(l.get("dram__bytes_read.sum", 0.0) + l.get("dram__bytes_write.sum", 0.0)
               for l in bwd)
    return dram, sum(l.get("lts__t_bytes.sum", 0.0) for l in bwd), [l["name"] for l in bwd]


def _summarize(paths):
    out = []
    for p in paths:
        if "_fused_" not in p:
            continue
        m = re.search(r"n(\d+)_d(\d+)", p)
        n, d = int(m.group(1)), int(m.group(2))
        fd, fl, _ = _bwd_bytes(p)
        mp = p.replace("_fused_", "_mat_")
        md, ml = (float("nan"), float("nan"))
        if mp in paths:
            md, ml, _ = _bwd_bytes(mp)
        row = {"n": n, "d": d, "fused_dram": fd, "fused_l2": fl, "mat_dram": md, "mat_l2": ml}
        elt = 2
        row["compulsory"] = B * H * (7 * n * d * elt + 2 * n * 4 + 2 * n * d * elt)
        bnk, bm = 128, (64 if d == 256 else 128)
        row["tile_m"] = bnk * d * 2            # K and V tiles resident per CTA (elements)
        row["n2d2_over_m"] = B * H * n * n * d * d / row["tile_m"] * elt
        out.append(row)
    out.sort(key=lambda r: (r["d"], r["n"]))
    print("| n | d | fused DRAM MB | fused L2<->SM MB | mat-P DRAM MB | mat-P L2<->SM MB | "
          "compulsory MB | n^2 d^2 / M MB (M = K,V tile) | fused L2 / (n^2 d^2 / M) |")
    print("|---|---|---|---|---|---|---|---|---|")
    for r in out:
        print("| %d | %d | %.1f | %.1f | %.1f | %.1f | %.1f | %.1f | %.2f |" % (
            r["n"], r["d"], r["fused_dram"] / 1e6, r["fused_l2"] / 1e6, r["mat_dram"] / 1e6,
            r["mat_l2"] / 1e6, r["compulsory"] / 1e6, r["n2d2_over_m"] / 1e6,
            r["fused_l2"] / r["n2d2_over_m"]))


def _keyrows(paths):
    """Key-tile kernel bytes per (n, d, R) from captures of that kernel alone."""
    out = []
    for p in paths:
        m = re.search(r"n(\d+)_d(\d+)_r(\d+)", p)
        n, d, r = (int(x) for x in m.groups())
        ls = [l for l in _rows(p) if l["name"].startswith("bwd_kv")]
        dram = sum(l.get("dram__bytes_read.sum", 0.0) + l.get("dram__bytes_write.sum", 0.0)
                   for l in ls)
        l2 = sum(l.get("lts__t_bytes.sum", 0.0) for l in ls)
        m_elems = 2 * r * d                       # K and V rows the CTA keeps
        ref = B * H * n * n * d * d / m_elems * 2  # n^2 d^2 / M words, in bf16 bytes
        out.append({"n": n, "d": d, "r": r, "M": m_elems, "dram": dram, "l2": l2, "ref": ref})
    out.sort(key=lambda x: (x["d"], x["n"], -x["r"]))
    base = {(x["n"], x["d"]): x["l2"] for x in out if x["r"] == 128}
    print("| n | d | key rows R | M = 2 R d | key-tile kernel L2<->SM MB | x vs R = 128 | "
          "DRAM MB | n^2 d^2 / M MB | L2 / (n^2 d^2 / M) |")
    print("|---|---|---|---|---|---|---|---|---|")
    for x in out:
        b0 = base.get((x["n"], x["d"]))
        print("| %d | %d | %d | %d | %.1f | %s | %.1f | %.1f | %.2f |" % (
            x["n"], x["d"], x["r"], x["M"], x["l2"] / 1e6,
            "%.2f" % (x["l2"] / b0) if b0 else "-", x["dram"] / 1e6, x["ref"] / 1e6,
            x["l2"] / x["ref"]))


def _sparse(paths):
    """Key-tile kernel bytes of the block-sparse backward against Theorem 4.5."""
    from .flops import kept_entries

    out = []
    for p in paths:
        m = re.search(r"n(\d+)_d(\d+)_w(\d+)g(\d+)r(\d+)", p)
        n, d, w_, g_, r_ = (int(x) for x in m.groups())
        mask = sparse_pattern(n, (w_, g_, r_)).numpy()
        z_qk = kept_entries(mask, n, False)
        ls = [l for l in _rows(p) if l["name"].startswith("bwd_kv")]
        dram = sum(l.get("dram__bytes_read.sum", 0.0) + l.get("dram__bytes_write.sum", 0.0)
                   for l in ls)
        l2 = sum(l.get("lts__t_bytes.sum", 0.0) for l in ls)
        z_in = n * d
        m_el = 256 * d                               # K and V tiles of a key-tile CTA
        out.append({"n": n, "d": d, "pat": (w_, g_, r_), "frac": mask.mean(), "zqk": z_qk,
                    "l2": l2, "dram": dram, "t1": z_in * z_in / m_el,
                    "t2": z_in * z_qk ** 0.5 / m_el ** 0.5, "split": z_in * z_in / z_qk,
                    "m": m_el})
    out.sort(key=lambda x: (x["d"], x["n"], x["zqk"]))
    print("| n | d | pattern (window, global, random) | blocks kept | Z_QK / n^2 | key-tile "
          "kernel L2<->SM MB (per head) | L2 bytes per kept entry | DRAM MB (per head) | "
          "Z_in^2/M MB | Z_in sqrt(Z_QK)/sqrt(M) MB | M = 256 d | split Z_in^2/Z_QK | regime |")
    print("|---|---|---|---|---|---|---|---|---|---|---|---|---|")
    for x in out:
        regime = "large cache" if x["m"] >= x["split"] else "small cache"
        print("| %d | %d | %s | %.1f %% | %.4f | %.1f | %.2f | %.2f | %.2f | %.2f | %d | %.0f | %s |"
              % (x["n"], x["d"], "%d, %d, %d" % x["pat"], 100 * x["frac"], x["zqk"] / x["n"] ** 2,
                 x["l2"] / H / 1e6, x["l2"] / H / x["zqk"], x["dram"] / H / 1e6,
                 2 * x["t1"] / 1e6, 2 * x["t2"] / 1e6, x["m"], x["split"], regime))


def _hbm_peak():
    p = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                     "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _kernels(path):
    peak, src = _hbm_peak()
    print("| # | kernel | time us | DRAM MB (read + write) | DRAM GB/s | of %s %.0f GB/s |"
          % (src, peak))
    print("|---|---|---|---|---|---|")
    for i, l in enumerate(_rows(path)):
        t = l.get("gpu__time_duration.sum", 0.0)   # ns
        rd = l.get("dram__bytes_read.sum", 0.0)
        wr = l.get("dram__bytes_write.sum", 0.0)
        gbs = (rd + wr) / t if t > 0 else 0.0        # bytes / ns = GB/s
        print("| %d | %s | %.1f | %.1f + %.1f | %.0f | %.1f %% |" % (
            i, l["name"], t / 1e3, rd / 1e6, wr / 1e6, gbs, 100.0 * gbs / peak))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    sub = ap.add_subparsers(dest="cmd", required=True)
    r = sub.add_parser("run")
    r.add_argument("--path", choices=["fused", "mat", "sparse"], required=True)
    r.add_argument("--pattern", default="2,1,2",
                   help="sparse: window, global and random blocks of the block pattern")
    r.add_argument("--n", type=int, required=True)
    r.add_argument("--d", type=int, required=True)
    r.add_argument("--B", type=int, default=B)
    r.add_argument("--H", type=int, default=H)
    r.add_argument("--causal", action="store_true")
    r.add_argument("--dtype", choices=["bf16", "f32"], default="bf16",
                   help="f32 runs the fp32 SIMT kernels (fused path only)")
    r.add_argument("--key-rows", type=int, default=0, choices=[0, 32, 64, 128],
                   help="fused bf16 backward with key tiles of this many keys (0: the product "
                        "kernels through attn_bwd)")
    tm = sub.add_parser("time")
    tm.add_argument("--path", choices=["fused", "mat"], required=True)
    tm.add_argument("--n", type=int, required=True)
    tm.add_argument("--d", type=int, required=True)
    tm.add_argument("--B", type=int, default=B)
    tm.add_argument("--H", type=int, default=H)
    tm.add_argument("--causal", action="store_true")
    kr = sub.add_parser("keyrows")
    kr.add_argument("csv", nargs="+")
    sp = sub.add_parser("sparse")
    sp.add_argument("csv", nargs="+")
    s = sub.add_parser("summarize")
    s.add_argument("csv", nargs="+")
    kk = sub.add_parser("kernels")
    kk.add_argument("csv")
    a = ap.parse_args(argv)
    if a.cmd == "run":
        _run(a.path, a.n, a.d, a.B, a.H, a.causal, a.dtype, a.key_rows,
             tuple(int(x) for x in a.pattern.split(",")))
    elif a.cmd == "time":
        _time(a.path, a.n, a.d, a.B, a.H, a.causal)
    elif a.cmd == "keyrows":
        _keyrows(a.csv)
    elif a.cmd == "sparse":
        _sparse(a.csv)
    elif a.cmd == "kernels":
        _kernels(a.csv)
    else:
        _summarize(a.csv)


if __name__ == "__main__":
    main(sys.argv[1:])
