"""GPU-vs-oracle comparison for the KDA step (test infrastructure).

The step has BF16 decision points (q, k, v after SiLU, the raw gate, o).  Two
correct FP32 implementations can round a value that lies within a few FP32 ulp
of a BF16 midpoint to different neighbours; the module docstring of the vLLM
page "...cutedsl.kda.wide" allows exactly that ("only FP32 reduction order
differs"), and the approximate exp/divide instructions add a few ulp more.
So the comparison is anchored:

Stage 1 (decision points): the GPU's BF16 q, k, v, raw_g (written through the
    library's ``dbg`` buffer by the same kernel) must equal the oracle's, or
    differ by exactly one BF16 ulp with the oracle's unrounded value within a
    band of the midpoint between the two candidates that the two sides'
    arithmetic errors allow:
      q, k, v:  |y - mid| <= silu_band(a) |y|, a = the SiLU argument (the
                conv sum, bit-identical on both sides: same FMA chain);
                silu_band is derived in its docstring from the error bounds of
                the instructions the kernel uses
      raw_g:    each side a correct BF16 rounding of a value within
                2 * 128 * 2^-24 * sum|products| of the exact float64 sum
    and differences must stay rare (at most ceil(1e-4 * elements)).
Stage 2 (everything else): the oracle re-run with the GPU's BF16 values forced
    in (teacher forcing) must match the GPU:
      state pool        |gpu - ora| <= 1e-5 + 1e-4 |ora| on every element;
                        pages no item writes are bit-identical to the input;
      output            within 2 BF16 ulp of max(|ora|, 2^-6) (outputs are
                        normalised to unit RMS); padded/error rows exactly +0;
      conv pool, rec_kg bit-exact;   rec_u  1e-5 + 1e-4 |ora|.
Unanchored (reported, not a gate): the GPU against the oracle's own result,
    with no forcing: BF16 flips, output ulps, state and rec_u error as a
    fraction of the tolerance and the count of elements beyond it.  This needs
    no ``dbg`` buffer, so it also covers launches without one (the
    configuration a caller runs); ``same_bits`` checks such a launch against a
    ``dbg`` launch of the same inputs bit for bit.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np
import torch

import oracle
from linear_attention_recurrent_kda_gb300.api import step_from_inputs
from tests.hostdata import bf16_bits_to_f64, bf16_ulp_diff, bits, to_oracle

GATE_BAND_ULPS = 2 * 128
FLIP_RATE_MAX = 1e-4
STATE_RTOL, STATE_ATOL = 1e-4, 1e-5
OUT_ULPS = 2
# The outputs are RMS-normalised (RMS ~ norm_weight * sigmoid(gate) <= 1.5);
# an element far below that scale carries the absolute FP32 error of the
# un-normalised recurrence output, so its ulps are counted at 2^-6.
OUT_FLOOR = 2.0 ** -6


def silu_band(a):
    """Relative band around the oracle's unrounded SiLU value y = a/(1+e^-a)
    inside which the kernel's value may fall on the other side of a BF16
    midpoint.  Kernel: e = ex2.approx(fl(-a * fl(log2 e))) (relative error
    <= 2^-22 for the instruction, plus |a| * 1.25 * 2^-24 from rounding the
    argument and the constant), den = fl(1 + e), y = div.full(a, den)
    (<= 2 ulp <= 2^-22).  Oracle: exp in double rounded once, then two
    correctly rounded operations (<= 3 * 2^-24).  The error of e enters y
    scaled by w = e / (1 + e).  First order, with one unit of slack:
        |y_gpu - y_ora| <= |y| 2^-24 (8 + w (6 + 1.25 |a|))."""
    a = np.asarray(a, np.float64)
    with np.errstate(over="ignore"):
        e = np.exp(-a)
        w = np.where(np.isinf(e), 1.0, e / (1.0 + e))
    return 2.0 ** -24 * (8.0 + w * (6.0 + 1.25 * np.abs(a)))


def bf16_ulp_at(v):
    v = np.asarray(v, np.float64)
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -126)))
    return np.exp2(e - 7)


def to_device(inputs: Dict[str, object], device="cuda") -> Dict[str, object]:
    out = {}
    for k, v in inputs.items():
        out[k] = v.to(device) if isinstance(v, torch.Tensor) else v
    return out


def run_gpu(inputs: Dict[str, object], *, dbg: bool = True, reps: int = 1,
            stream: Optional[torch.cuda.Stream] = None, path: int = 0,
            balance: bool = True, noalloc: bool = False) -> Dict[str, object]:
    """One step of the CUDA library on a device copy of ``inputs`` (``balance``:
    the step's own scheduler words, as the binding sets by default, or fixed
    contiguous ranges only; ``noalloc``: through kda_step_noalloc, the
    library's own words)."""
    d = to_device(inputs)
    B, H, T = d["batch"], d["heads"], d["tokens"]
    dev = torch.device("cuda")
    out = torch.full((B * T, H * 128), float("nan"), dtype=torch.bfloat16, device=dev)
    rec_u = rec_kg = None
    if d["record"]:
        rec_u = torch.zeros((B, H, T, 128), dtype=torch.float32, device=dev)
        rec_kg = torch.zeros((B, H, T, 256), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    dbgt = (torch.zeros((B, H, T, 4, 128), dtype=torch.bfloat16, device=dev)
            if dbg else None)
    step = step_from_inputs(d, out, rec_u=rec_u, rec_kg=rec_kg, err=err, dbg=dbgt,
                            path=path, balance=balance, noalloc=noalloc)
    if stream is not None:
        stream.wait_stream(torch.cuda.current_stream())
    for _ in range(reps):
        step(stream)
    torch.cuda.synchronize()
    res = {"output": bits(out), "state": d["state"].cpu().numpy(),
           "conv_state": bits(d["conv_state"]), "err": int(err.item())}
    if d["record"]:
        res["rec_u"] = rec_u.cpu().numpy()
        res["rec_kg"] = bits(rec_kg)
    if dbg:
        res["dbg"] = bits(dbgt)
    return res


def live_items(o: Dict[str, object]) -> np.ndarray:
    """Items (r*H + h) whose request resolves to a valid live slot."""
    B, H, T, ns = o["batch"], o["heads"], o["tokens"], o["num_slots"]
    live = np.zeros(B, bool)
    for r in range(B):
        if T == 1:
            s = int(o["slots"][r]); cs = s
        else:
            a = int(o["accepted"][r])
            if not 1 <= a <= T:
                continue
            s = int(o["slots"][r, a - 1]); cs = int(o["slots"][r, 0])
        if s <= 0 or s >= ns or cs <= 0 or cs >= ns:
            continue
        if T > 1 and not o["record"] and (o["slots"][r, :T] >= ns).any():
            continue
        live[r] = True
    return np.array([r * H + h for r in range(B) if live[r] for h in range(H)], np.int64)


def written_pages(o: Dict[str, object], items: Sequence[int]):
    """(slot, head) pages the listed live items write."""
    H, T = o["heads"], o["tokens"]
    pages = set()
    if o["record"]:
        return pages
    for it in items:
        r, h = divmod(int(it), H)
        if T == 1:
            pages.add((int(o["slots"][r]), h))
        else:
            for t in range(T):
                s = int(o["slots"][r, t])
                if s > 0:
                    pages.add((s, h))
    return pages


def stage1(o, gpu_dbg, ora, items) -> Dict[str, int]:
    """Decision-point check; returns flip counts.

    q, k, v: the SiLU inputs are bit-identical on both sides (same FMA chain),
    so a BF16 value may differ only by one ulp, at a midpoint the oracle's
    unrounded value lies within silu_band(a) of.  raw_g: the FP32 gate sum has an
    absolute error bound (2 * 128 * 2^-24 * sum|products|), which near zero can
    span several BF16 ulps, so each side's BF16 raw gate must be a correct
    rounding of some value within that bound of the exact (float64) sum."""
    B, H, T, D = o["batch"], o["heads"], o["tokens"], 128
    rs, hs = np.divmod(np.asarray(items, np.int64), H)
    g = gpu_dbg[rs, hs]                        # [n, T, 4, D]
    w = ora["inter"][rs, hs]
    pre = ora["pre"][rs, hs]
    sin = ora["silu_in"][rs, hs]
    ulps = bf16_ulp_diff(g, w)
    qkv = ulps[:, :, :3]
    assert qkv.max(initial=0) <= 1, f"BF16 q/k/v differ by {qkv.max()} ulp"
    gv, wv = bf16_bits_to_f64(g), bf16_bits_to_f64(w)
    counts = {"q": 0, "k": 0, "v": 0, "g": 0}
    for (n, t, part, c) in np.argwhere(qkv == 1):
        mid = 0.5 * (gv[n, t, part, c] + wv[n, t, part, c])
        counts["qkv"[part]] += 1
        y = pre[n, t, part, c]
        a = sin[n, t, part, c]
        assert abs(y - mid) <= silu_band(a) * abs(y), (
            f"SiLU flip outside band: item {rs[n]*H+hs[n]} t{t} part{part} c{c} "
            f"a={a!r} y={y!r} mid={mid!r} band={silu_band(a)!r}")
    # gate: exact sums of the sampled (item, token, feature) triples
    fa = bf16_bits_to_f64(o["f_a"])
    fb = bf16_bits_to_f64(o["f_b"]).reshape(H, D, -1)
    rows = (rs[:, None] * T + np.arange(T)[None, :])          # [n, T]
    fa_rows = fa[rows]                                         # [n, T, R]
    fb_h = fb[hs]                                              # [n, D, R]
    exact = np.einsum("ntr,nfr->ntf", fa_rows, fb_h)
    mag = np.einsum("ntr,nfr->ntf", np.abs(fa_rows), np.abs(fb_h))
    band = GATE_BAND_ULPS * 2.0 ** -24 * mag
    for side, vals in (("gpu", gv[:, :, 3]), ("oracle", wv[:, :, 3])):
        half = 0.5 * bf16_ulp_at(np.abs(vals))
        ok = np.abs(vals - exact) <= band + half
        if not ok.all():
            n, t, f = np.argwhere(~ok)[0]
            raise AssertionError(
                f"{side} raw gate not a rounding of the exact sum: item "
                f"{rs[n]*H+hs[n]} t{t} f{f}: {vals[n, t, f]!r} exact "
                f"{exact[n, t, f]!r} band {band[n, t, f]!r}")
    counts["g"] = int((ulps[:, :, 3] > 0).sum())
    flips = int((ulps > 0).sum())
    total = g.size
    assert flips <= int(np.ceil(FLIP_RATE_MAX * total)), f"{flips} flips of {total}"
    counts["flips"] = flips
    counts["total"] = int(total)
    return counts


def compare(inputs: Dict[str, object], gpu: Dict[str, object],
            items: Optional[Sequence[int]] = None) -> Dict[str, object]:
    """Anchored comparison of one GPU step with the oracle.

    ``items`` restricts the oracle to a sample of items (full-size runs); the
    checks then cover those items' outputs and pages only."""
    o = to_oracle(inputs)
    B, H, T = o["batch"], o["heads"], o["tokens"]
    dim = H * 128
    live = live_items(o)
    sample = live if items is None else np.intersect1d(np.asarray(items), live)
    ora = oracle.run(o, mode="f32", items=None if items is None else items,
                     want_intermediates=True)
    stats = stage1(o, gpu["dbg"], ora, sample) if len(sample) else {}

    forced = np.zeros_like(ora["inter"])
    if len(sample):
        rs, hs = np.divmod(sample, H)
        forced[rs, hs] = gpu["dbg"][rs, hs]
    tf = oracle.run(o, mode="f32", items=None if items is None else items,
                    forced=forced)

    sel_items = np.arange(B * H) if items is None else np.asarray(items)
    rows = []
    for it in sel_items:
        r, h = divmod(int(it), H)
        for t in range(T):
            rows.append(((r * T + t), h))
    rr = np.array([x[0] for x in rows]); hh = np.array([x[1] for x in rows])
    cols = hh[:, None] * 128 + np.arange(128)[None, :]
    g_out = gpu["output"][rr[:, None], cols]
    t_out = tf["output"][rr[:, None], cols]
    d = bf16_ulp_diff(g_out, t_out)
    gf, tfv = bf16_bits_to_f64(g_out), bf16_bits_to_f64(t_out)
    tol = OUT_ULPS * bf16_ulp_at(np.maximum(np.abs(tfv), OUT_FLOOR))
    bad = np.argwhere(~(np.abs(gf - tfv) <= tol))
    if len(bad):
        i, c = bad[0]
        raise AssertionError(
            f"{len(bad)} output elements beyond {OUT_ULPS} BF16 ulp (floor "
            f"{OUT_FLOOR}); first: row {rr[i]} head {hh[i]} chan {c}: gpu "
            f"{gf[i, c]!r} oracle {tfv[i, c]!r} ({d[i, c]} ulp)")
    stats["out_max_ulp"] = int(d.max(initial=0))
    stats["out_exact_frac"] = float((d == 0).mean()) if d.size else 1.0

    # padded / error items: exact zeros
    live_set = set(int(x) for x in live)
    for it in sel_items:
        if int(it) in live_set:
            continue
        r, h = divmod(int(it), H)
        blk = gpu["output"][r * T:(r + 1) * T, h * 128:(h + 1) * 128]
        assert not blk.any(), f"padded item {it} output not +0"

    # state: written pages within tolerance, others bit-identical to input
    wp = written_pages(o, sample)
    st_in = o["state"]
    worst = 0.0
    if items is None:
        pages = [(s, h) for s in range(o["num_slots"]) for h in range(H)]
    else:
        pages = sorted(wp | {(int(o["slots"][int(i) // H] if T == 1 else
                                 o["slots"][int(i) // H, 0]), int(i) % H)
                             for i in sel_items})
    for (s, h) in pages:
        if s <= 0 or s >= o["num_slots"]:
            continue
        gp, tp = gpu["state"][s, h], tf["state"][s, h]
        if (s, h) in wp:
            err = np.abs(gp.astype(np.float64) - tp)
            lim = STATE_ATOL + STATE_RTOL * np.abs(tp)
            assert np.all(err <= lim), (
                f"state page ({s},{h}) off by {float((err - lim).max())} over tol")
            worst = max(worst, float((err / lim).max()))
        else:
            assert np.array_equal(gp.view(np.uint32), st_in[s, h].view(np.uint32)), (
                f"untouched page ({s},{h}) changed")
    stats["state_worst_frac_of_tol"] = worst

    # conv pool: bit-exact on the sampled items' rows (all rows when full)
    if items is None:
        assert np.array_equal(gpu["conv_state"], tf["conv_state"]), "conv state"
    else:
        for it in sel_items:
            r, h = divmod(int(it), H)
            cs = int(o["slots"][r]) if T == 1 else int(o["slots"][r, 0])
            if cs <= 0 or cs >= o["num_slots"]:
                continue
            for p in range(3):
                ch = slice(p * dim + h * 128, p * dim + (h + 1) * 128)
                assert np.array_equal(gpu["conv_state"][cs, ch], tf["conv_state"][cs, ch]), (
                    f"conv rows of item {it}")

    if o["record"]:
        rs, hs = np.divmod(np.asarray(sel_items), H)
        assert np.array_equal(gpu["rec_kg"][rs, hs], tf["rec_kg"][rs, hs]), "rec_kg"
        gu, tu = gpu["rec_u"][rs, hs], tf["rec_u"][rs, hs]
        assert np.all(np.abs(gu - tu) <= STATE_ATOL + STATE_RTOL * np.abs(tu)), "rec_u"

    assert gpu["err"] == tf["err"], f"error word {gpu['err']} != {tf['err']}"

    # unanchored (reported, not a gate)
    stats.update(unanchored(inputs, gpu, items=items, ora=ora, o=o))
    return stats


def unanchored(inputs: Dict[str, object], gpu: Dict[str, object],
               items: Optional[Sequence[int]] = None, ora=None, o=None) -> Dict[str, object]:
    """The GPU result against the oracle's own (no teacher forcing): a report,
    not a gate.  Needs no ``dbg`` buffer.  BF16 flips of the intermediates are
    counted when the GPU result carries them; outputs in BF16 ulps; written
    state pages and rec_u as the worst error over the anchored tolerance
    1e-5 + 1e-4 |ora| and the number of elements beyond it (a flipped raw
    gate moves its key's decay by up to about 1.5 %, so these can exceed the
    tolerance without either side being wrong)."""
    if o is None:
        o = to_oracle(inputs)
    H, T = o["heads"], o["tokens"]
    sel = np.arange(o["batch"] * H) if items is None else np.asarray(items, np.int64)
    if ora is None:
        ora = oracle.run(o, mode="f32", items=None if items is None else sel,
                         want_intermediates="dbg" in gpu)
    rep: Dict[str, object] = {}
    rs, hs = np.divmod(sel, H)
    if "dbg" in gpu:
        live = np.intersect1d(sel, live_items(o))
        lr, lh = np.divmod(live, H)
        fl = bf16_ulp_diff(gpu["dbg"][lr, lh], ora["inter"][lr, lh]) > 0
        rep["unanchored_flips"] = {"qkv": int(fl[:, :, :3].sum()),
                                   "g": int(fl[:, :, 3].sum()), "total": int(fl.size)}
    rows = (rs[:, None] * T + np.arange(T)[None, :]).reshape(-1)
    heads = np.repeat(hs, T)
    cols = heads[:, None] * 128 + np.arange(128)[None, :]
    ud = bf16_ulp_diff(gpu["output"][rows[:, None], cols], ora["output"][rows[:, None], cols])
    rep["unanchored_out_max_ulp"] = int(ud.max(initial=0))
    rep["unanchored_out_beyond_2ulp"] = int((ud > OUT_ULPS).sum())
    worst, beyond, maxabs = 0.0, 0, 0.0
    for (s, h) in sorted(written_pages(o, np.intersect1d(sel, live_items(o)))):
        if s <= 0 or s >= o["num_slots"]:
            continue
        ref = ora["state"][s, h].astype(np.float64)
        err = np.abs(gpu["state"][s, h].astype(np.float64) - ref)
        lim = STATE_ATOL + STATE_RTOL * np.abs(ref)
        worst = max(worst, float((err / lim).max()))
        beyond += int((err > lim).sum())
        maxabs = max(maxabs, float(err.max()))
    rep["unanchored_state_worst_frac_of_tol"] = worst
    rep["unanchored_state_beyond_tol"] = beyond
    rep["unanchored_state_max_abs"] = maxabs
    if o["record"]:
        gu, tu = gpu["rec_u"][rs, hs].astype(np.float64), ora["rec_u"][rs, hs]
        lim = STATE_ATOL + STATE_RTOL * np.abs(tu)
        e = np.abs(gu - tu)
        rep["unanchored_rec_u_worst_frac_of_tol"] = float((e / lim).max(initial=0.0))
        rep["unanchored_rec_u_beyond_tol"] = int((e > lim).sum())
    return rep


def same_bits(a: Dict[str, object], b: Dict[str, object]) -> None:
    """Two GPU results of the same inputs are identical bit for bit: outputs,
    both pools, records and the error word (the ``dbg`` dump is compared only
    when both carry it)."""
    for key in ("output", "state", "conv_state", "rec_u", "rec_kg", "dbg"):
        if key in a and key in b:
            x, y = np.asarray(a[key]), np.asarray(b[key])
            assert x.shape == y.shape and np.array_equal(x.view(np.uint8), y.view(np.uint8)), (
                f"{key} differs between the two launches")
    assert a["err"] == b["err"], f"error word {a['err']} != {b['err']}"
