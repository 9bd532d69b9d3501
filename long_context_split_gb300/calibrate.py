"""Calibrate the critical-wave split model on this GPU (LiquidCP Appendix A.2,
"Calibration": fit the time unit, rho and delta_attn to measured busy
times, then delta_red and gamma).

The planner scores a split plan with the critical-wave model (LiquidCP
Section 5.2, Eqs. 5-6): attention tasks of n_t tiles plus a fixed
delta_attn, run on K scheduling units at a rate set by tau(k) =
max(rho, k/K), then reductions of cost delta_red + gamma * v * s on the
released warps.  The constants the pages print (Table 2) were fitted on
H100 for LiquidCP's engine.  This script measures this library's kernels on
seeded calibration batches of mixed lengths and split counts (kernel device
time from the launch profiler), grid-searches (rho, delta_attn, delta_red,
gamma) with the least-squares time unit for each candidate, and keeps the
candidate with the lowest relative RMS error between unit * model score and
the measured time.

    python -m long_context_split_gb300.calibrate            # both kernels
    python -m long_context_split_gb300.calibrate --path mla

It writes ``csrc/calibration.h`` (the constants the library uses for plans
whose model parameters are left at their defaults) and ``calibration.json``
(the batches, measurements and fit); rebuild the library afterwards.
Needs a GPU; takes a few minutes.
"""
from __future__ import annotations

import argparse
import datetime
import itertools
import json
import os
import sys

import numpy as np

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# search grid
RHO = [0.05, 0.1, 0.15, 0.2, 0.3, 0.43, 0.6, 0.8, 1.0]
DELTA_ATTN = [0.0, 1.0, 2.0, 4.0, 8.0, 16.0, 32.0, 64.0]
DELTA_RED = [0.0, 1.0, 2.5, 5.0, 10.0, 20.0]
GAMMA = [0.0, 0.1, 0.25, 0.47, 1.0, 2.0]
SPLITS = [1, 2, 4, 8, 16]

# (name, base configuration, batch recipe)
PATHS = {
    "gqa": ("llama405b_gqa_decode", "gqa_engine_kernel"),
    "mla": ("deepseek_mla_decode", "mla_partial_kernel"),
}


def _lengths(rng, recipe):
    kind, b = recipe[0], recipe[1]
    if kind == "const":
        return np.full(b, recipe[2], dtype=np.int64)
    if kind == "uniform":
        return rng.integers(recipe[2], recipe[3], size=b)
    if kind == "loguniform":
        return np.exp(rng.uniform(np.log(recipe[2]), np.log(recipe[3]), size=b)).astype(np.int64)
    if kind == "skewed":      # a few long histories among many short ones
        return np.array([recipe[2]] * recipe[3] + [recipe[4]] * (b - recipe[3]), dtype=np.int64)
    raise ValueError(kind)


RECIPES = [
    ("const", 16, 32768),
    ("const", 4, 131072),
    ("uniform", 32, 1024, 65536),
    ("loguniform", 16, 1024, 131072),
    ("loguniform", 64, 1024, 131072),
    ("skewed", 32, 131072, 4, 2048),
]


def _model_seq(spec, L, q_len=1):
    """(tiles, tasks per split, output vectors, q_len) as the library's planner builds them for
    decode requests: one tile per page, one row block per KV head (GQA) or one task per token (MLA)."""
    tiles = -(-int(L) // spec.page_size)
    tasks = spec.num_kv_heads if spec.kind == "gqa" else 1
    return (tiles, tasks, q_len * spec.num_q_heads, q_len)


def measure(path: str, reps: int = 10, seed: int = 7):
    """Measured device time (ms) of each calibration batch and split count."""
    import dataclasses
    import torch
    import long_context_split_gb300 as skv
    import workloads as W
    base, kernel = PATHS[path]
    rng = np.random.default_rng(seed)
    samples = []
    for ri, recipe in enumerate(RECIPES):
        L = np.maximum(_lengths(rng, recipe), 64)
        spec = dataclasses.replace(W.get_config(base), batch=len(L), seed=100 + ri)
        wl = W.build_workload(spec, seq_lens=L.astype(np.int32))
        t = wl.device_tensors("cuda")
        prob = skv.AttentionProblem(
            q=t["q"], k_cache=t["k"], v_cache=t["v"], page_table=t["page_table"], seq_lens=t["seq_lens"],
            qo_indptr=t["qo_indptr"], num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
            head_dim_qk=spec.head_dim_qk, head_dim_v=spec.head_dim_v, page_size=spec.page_size,
            scale=spec.scale, kind=spec.kind, seq_lens_host=wl.seq_lens, qo_indptr_host=wl.qo_indptr)
        for sp in SPLITS:
            att = skv.SplitKVAttention(prob, skv.plan_params("uniform", uniform_splits=sp))
            for _ in range(2):
                att.decode()
            torch.cuda.synchronize()
            skv.profile_begin()
            for _ in range(reps):
                att.decode()
            torch.cuda.synchronize()
            k = skv.profile_end()
            att.check_device_error()
            ms = sum(v[1] for v in k.values()) / reps
            samples.append({"recipe": list(recipe), "lengths": [int(x) for x in L], "splits": sp, "ms": ms,
                            "kernel_ms": {n: v[1] / reps for n, v in k.items()}})
            print(f"{path} batch {ri} {recipe[0]:10s} B={len(L):3d} splits {sp:2d}: {ms:.4f} ms", flush=True)
        del t, prob
        torch.cuda.empty_cache()
    return spec_for(path), samples


def spec_for(path: str):
    import workloads as W
    return W.get_config(PATHS[path][0])


def fit(path: str, spec, samples, num_ctas: int, warps: int):
    """Grid search; returns the best (params, unit_ms, rel_rmse) and per-sample predictions."""
    import long_context_split_gb300 as skv
    seqs = [[_model_seq(spec, L) for L in s["lengths"]] for s in samples]
    t = np.array([s["ms"] for s in samples])
    best = None
    for rho, da, dr, g in itertools.product(RHO, DELTA_ATTN, DELTA_RED, GAMMA):
        sc = np.array([skv.model_simulate(sq, [s["splits"]] * len(sq), num_ctas=num_ctas, warps_per_cta=warps,
                                          q_heads=spec.num_q_heads, rho=rho, delta_attn=da, delta_red=dr,
                                          gamma=g)[0] for sq, s in zip(seqs, samples)])
        r = sc / t
        unit = float(np.sum(r) / np.sum(r * r))      # least squares of (unit * score - t) / t
        err = float(np.sqrt(np.mean((unit * r - 1.0) ** 2)))
        if best is None or err < best[2]:
            best = ((rho, da, dr, g), unit, err, sc)
    (rho, da, dr, g), unit, err, sc = best
    return {"rho": rho, "delta_attn": da, "delta_red": dr, "gamma": g, "unit_ms": unit, "rel_rmse": err,
            "num_ctas": num_ctas, "warps_per_cta": warps,
            "predicted_ms": [float(unit * x) for x in sc]}


def write_header(fits: dict, when: str, gpu: str):
    def line(name, f):
        return (f"constexpr Fit {name} = {{{f['rho']}, {f['delta_attn']}, {f['delta_red']}, {f['gamma']}}};"
                f"   // time unit {1e3 * f['unit_ms']:.3f} us per tile-equivalent, relative RMS error "
                f"{100 * f['rel_rmse']:.1f} %")
    table2 = {"rho": 0.43, "delta_attn": 32.0, "delta_red": 2.5, "gamma": 0.47}
    gqa = fits.get("gqa")
    mla = fits.get("mla")
    text = f"""// Critical-wave model constants used when a plan leaves the model parameters
// at their defaults (LiquidCP Section 5.2, Eqs. 5-6; Appendix A.2
// "Calibration").  Written by long_context_split_gb300/calibrate.py on {when}
// ({gpu}); a kernel without a fit keeps LiquidCP Table 2's H100 values.
#pragma once

namespace skv {{
namespace calib {{

struct Fit {{
    double rho, delta_attn, delta_red, gamma;
}};

{line("kGqaEngine", gqa) if gqa else "constexpr Fit kGqaEngine = {0.43, 32.0, 2.5, 0.47};   // LiquidCP Table 2"}
{line("kMla", mla) if mla else "constexpr Fit kMla = {0.43, 32.0, 2.5, 0.47};   // LiquidCP Table 2"}
constexpr Fit kTable2 = {{{table2['rho']}, {table2['delta_attn']}, {table2['delta_red']}, {table2['gamma']}}};

}}  // namespace calib
}}  // namespace skv
"""
    with open(os.path.join(PKG, "csrc", "calibration.h"), "w") as f:
        f.write(text)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--path", choices=["gqa", "mla", "both"], default="both")
    ap.add_argument("--reps", type=int, default=10)
    args = ap.parse_args()
    import torch
    import long_context_split_gb300 as skv  # noqa: F401
    jpath = os.path.join(PKG, "calibration.json")
    record = json.load(open(jpath)) if os.path.exists(jpath) else {}
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    gpu = torch.cuda.get_device_name(0)
    paths = ["gqa", "mla"] if args.path == "both" else [args.path]
    for p in paths:
        spec, samples = measure(p, args.reps)
        # scheduling units and reduction warps of the kernel (the library's defaults)
        K, warps = (sms, 7) if p == "gqa" else (sms // 2, 1)
        f = fit(p, spec, samples, K, warps)
        print(f"{p}: rho {f['rho']} delta_attn {f['delta_attn']} delta_red {f['delta_red']} gamma {f['gamma']} "
              f"unit {1e3 * f['unit_ms']:.3f} us  rel RMSE {100 * f['rel_rmse']:.1f} %", flush=True)
        record[p] = {"fit": f, "samples": samples, "gpu": gpu}
    when = datetime.date.today().isoformat()
    record["when"] = when
    with open(jpath, "w") as fh:
        json.dump(record, fh, indent=1)
    fits = {p: record[p]["fit"] for p in ("gqa", "mla") if p in record}
    write_header(fits, when, gpu)
    print("wrote", jpath, "and csrc/calibration.h; rebuild the library to use them")


if __name__ == "__main__":
    main()
