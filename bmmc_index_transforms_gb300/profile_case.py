"""Run one permutation configuration a few times, for profilers.

    python -m bmmc_index_transforms_gb300.profile_case --kind random --n 26 --reps 3
    python -m bmmc_index_transforms_gb300.profile_case --kind lmad_slice_2d --shape 8192,8193 --reps 2

Kinds: random (seed), worst (seed, low 10 bits mapped to high bits), bitrev,
complement (A = I, c on the high bits: contiguous tiles on both sides),
window (seed, a random BMMC on the low --window bits and the identity above:
tiles scattered only inside aligned windows of 2^window elements),
transpose (square, n even), dims5 (the 5-D (4,2,0,3,1) permutation of a
[32,64,64,64,32]-shaped array scaled to n bits), copy (the copy kernel on the
same bytes), two_factor (seed, two passes through caller scratch).
General LMAD copies (--shape, --elem): lmad_slice_2d, lmad_slice_3d,
lmad_reversed_rows (the Futhark copy post's "Impact" functions on a
row-major array of that shape), lmad_transpose (the shape's axes
reversed, made contiguous) and lmad_permute (the shape's axes in the order
--perm, out dimension k = in dimension perm[k], made contiguous; --blocked
auto / force / never chooses for the blocked copy).
Prints the plan and the CUDA-event time of each repetition.
"""

from __future__ import annotations

import argparse
import sys

import torch

import bmmc_index_transforms_gb300 as bm
from bmmc_index_transforms_gb300 import maps, synth


def _accept(n, elem):
    def f(rows):
        try:
            bm.bmmc_plan_destroy(bm.bmmc_plan(n, rows, 0, elem))
            return True
        except bm.BmmcError as e:
            if e.status == 2:
                return False
            raise
    return f


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--kind", default="random",
                    choices=["random", "worst", "bitrev", "transpose", "dims5", "copy", "two_factor",
                             "complement", "window", "lmad_slice_2d", "lmad_slice_3d", "lmad_reversed_rows",
                             "lmad_transpose", "lmad_permute"])
    ap.add_argument("--n", type=int, default=26)
    ap.add_argument("--elem", type=int, default=4)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--t-in", type=int, default=0)
    ap.add_argument("--t-out", type=int, default=0)
    ap.add_argument("--tile-bits", type=int, default=0)
    ap.add_argument("--shape", default="8192,8193")
    ap.add_argument("--window", type=int, default=22, help="window: log2 elements of a window")
    ap.add_argument("--perm", default="", help="lmad_permute: axis order of the destination")
    ap.add_argument("--blocked", default="auto", choices=["auto", "force", "never"])
    a = ap.parse_args(argv)
    if a.kind.startswith("lmad_"):
        return lmad_case(a)
    n, elem = a.n, a.elem
    nbytes = (1 << n) * elem
    d_in = torch.arange(nbytes // 4, dtype=torch.int32, device="cuda")
    d_out = torch.empty_like(d_in)
    mode = 1 if a.kind == "two_factor" else 0
    if a.kind in ("random", "two_factor"):
        rows, c, _ = synth.draw_bmmc(a.seed, n, _accept(n, elem))
    elif a.kind == "worst":
        rows, c, _ = synth.draw_bmmc(a.seed, n, _accept(n, elem), low_to_high=min(10, n // 2))
    elif a.kind == "window":
        m = min(a.window, n)
        low, cl, _ = synth.draw_bmmc(a.seed, m, _accept(m, elem))
        rows, c = list(low) + maps.identity_rows(n)[m:], cl
    elif a.kind == "complement":
        # A = I, c on the bits above the tile: every tile is contiguous on both sides
        rows, c = maps.identity_rows(n), ((1 << n) - 1) & ~((1 << 16) - 1)
    elif a.kind == "bitrev":
        rows, c = maps.bitrev_rows(n), 0
    elif a.kind == "transpose":
        rows, c = maps.rotate_rows(n, n // 2), 0
    elif a.kind == "dims5":
        # split n bits like [32,64,64,64,32] (5,6,6,6,5 bits) scaled to n
        base = [5, 6, 6, 6, 5]
        while sum(base) > n:
            base[base.index(max(base))] -= 1
        while sum(base) < n:
            base[base.index(min(base))] += 1
        rows, c = maps.axes_rows(base, synth.FIVE_D_AXES), 0
    else:
        rows, c = None, 0
    stream = torch.cuda.current_stream()
    if rows is None:
        fn = lambda: bm.bmmc_copy(d_in, d_out, nbytes, stream)  # noqa: E731
        print(f"copy of {nbytes} bytes")
        plan = None
    else:
        plan = bm.Plan(rows, c, elem, mode=mode, t_in=a.t_in, t_out=a.t_out, tile_bits=a.tile_bits)
        print("plan:", plan.info)
        if mode == 1:
            scratch = torch.empty_like(d_in)
            fn = lambda: plan.permute_scratch(d_in, d_out, scratch, stream)  # noqa: E731
        else:
            fn = lambda: plan.permute(d_in, d_out, stream)  # noqa: E731
    for r in range(a.reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        torch.cuda.synchronize()
        ms = s.elapsed_time(e)
        print(f"rep {r}: {ms:.4f} ms, {2 * nbytes / ms / 1e6:.1f} GB/s effective")
    if plan:
        plan.close()
    return 0


def lmad_view(a) -> dict:
    """The LMAD copy of an lmad_* kind: sizes, offsets and strides in
    elements, as lmad_copy takes them."""
    shape = [int(v) for v in a.shape.split(",")]
    if a.kind in ("lmad_transpose", "lmad_permute"):
        perm = ([int(v) for v in a.perm.split(",")] if a.kind == "lmad_permute"
                else list(range(len(shape)))[::-1])
        if sorted(perm) != list(range(len(shape))):
            raise SystemExit("--perm must order the axes of --shape")
        out_rm = synth.row_major_strides([shape[p] for p in perm])
        out_strides = [0] * len(shape)
        for pos, p in enumerate(perm):
            out_strides[p] = out_rm[pos]
        total = 1
        for v in shape:
            total *= v
        return dict(sizes=shape, in_offset=0, in_strides=synth.row_major_strides(shape), in_elems=total,
                    out_offset=0, out_strides=out_strides, out_elems=total)
    return synth.page_lmad_workload(a.kind[len("lmad_"):], shape)


def lmad_case(a):
    e = a.elem
    w = lmad_view(a)
    src = torch.empty(w["in_elems"] * e, dtype=torch.uint8, device="cuda")
    dst = torch.empty(w["out_elems"] * e, dtype=torch.uint8, device="cuda")
    args = (w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], e)
    print("analysis:", bm.lmad_copy_query(*args, src, dst, blocked=a.blocked))
    stream = torch.cuda.current_stream()
    for r in range(a.reps):
        s, t = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        bm.lmad_copy(*args, src, dst, stream, blocked=a.blocked)
        t.record(stream)
        torch.cuda.synchronize()
        ms = s.elapsed_time(t)
        print(f"rep {r}: {ms:.4f} ms, {2 * w['out_elems'] * e / ms / 1e6:.1f} GB/s effective")
    return 0


if __name__ == "__main__":
    sys.exit(main())
