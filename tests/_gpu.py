"""GPU runners for the parity tests: each runs one C-ABI call through the binding on the
seeded inputs of a ``workloads`` case and returns the outputs as CPU tensors.  Plus the
tolerance rule shared by the tests.

Tolerance of the floating-point outputs:
  * fp32 I/O: max |x - ref| <= 1e-4.
  * bf16 I/O with fp32 arithmetic, "within 2e-2 relative to the per-tensor RMS":
      RMS(x - ref) <= 2e-2 * RMS(ref)                  over the compared tensor, and, per element,
      |x - ref|    <= 2e-2 * RMS(ref) + own(ref)
    where own(ref) = 2^-8 * |ref| for a result the kernel stores in bf16 and 0 for one it stores
    in fp32 (TreeWY's pseudo-values and log gamma).  The oracle's reference is the unrounded
    fp64 value, and a bf16 result is the kernel's fp32 value rounded once to nearest: with 8
    significant bits that one rounding moves it by at most half an ulp, 2^-8 of its magnitude.
    own(ref) is that one rounding and nothing more; every other error must fit in 2e-2 * RMS.
    Where the reference is itself a bf16 result of the library (two kernels compared with each
    other), each side carries its own rounding: own(ref) = 2 * 2^-8 * |ref|.
  * Attention outputs are compared twice (assert_attention_close): with the oracle whose rotated
    query is rounded to bf16 -- the operand precision of the tensor-core score product -- under
    the rule above, and with the plain fp64 oracle under the rule above plus, per element, the
    change that this one rounding makes to the oracle's own result.
Integer outputs are compared exactly.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import tree_speculative_verification_gdn_gb300 as tv
import workloads as W

DEV = "cuda"


def to_dev(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().to(DEV)


BF16_REL = 2e-2
BF16_OWN = 2.0 ** -8   # one round-to-nearest of a bf16-stored result

# One line per compared tensor: the margins of the comparison, collected for the terminal
# summary (conftest) and, when TV_PARITY_MARGINS names a file, written there as JSON lines.
MARGINS: list[dict] = []


def rms(x: np.ndarray) -> float:
    x = np.asarray(x, dtype=np.float64)
    return float(np.sqrt(np.mean(x * x))) if x.size else 0.0


def max_err(got, ref) -> float:
    g = W.f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    return float(np.abs(g - np.asarray(ref, dtype=np.float64)).max())


def _record(what: str, io: str, own: bool, g: np.ndarray, r: np.ndarray, diff: np.ndarray, own_k: float,
            extra=0.0) -> dict:
    scale = rms(r)
    m = dict(what=what, io=io, stored_bf16=own, own_k=own_k, n=int(r.size), rms_ref=scale, max_abs=float(diff.max()))
    if io != "f32" and scale > 0:
        strict = BF16_REL * scale
        m.update(max_over_rms=float(diff.max()) / scale, rms_err_over_rms=rms(g - r) / scale,
                 n_over_strict=int((diff > strict).sum()),
                 worst_vs_bound=float((diff / (strict + (own_k * np.abs(r) if own else 0.0) + extra)).max()))
    MARGINS.append(m)
    path = os.environ.get("TV_PARITY_MARGINS")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(m) + "\n")
    return m


def assert_close(got, ref, io: str, what: str, stored: str | None = None, ref_rounded: bool = False,
                 extra=None) -> None:
    """``io``: the workload's I/O type ("f32" or "bf16"), which picks the rule above.
    ``stored``: how the kernel stored the compared values ("bf16" or "f32"); taken from the
    tensor's dtype when ``got`` is a torch tensor, and required for numpy input under bf16 I/O.
    ``ref_rounded``: the reference is another kernel's bf16 result (two roundings allowed).
    ``extra``: a per-element allowance added to the bf16 bound (see assert_attention_close)."""
    if isinstance(got, torch.Tensor):
        st = "bf16" if got.dtype == torch.bfloat16 else "f32"
        assert stored in (None, st), f"{what}: stored={stored} but the tensor is {got.dtype}"
        stored = st
        g = W.f64(got)
    else:
        g = np.asarray(got, dtype=np.float64)
        assert io == "f32" or stored in ("bf16", "f32"), f"{what}: say how numpy input was stored"
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, f"{what}: shape {g.shape} vs {r.shape}"
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    if not g.size:
        return
    diff = np.abs(g - r)
    own = stored == "bf16"
    own_k = (2.0 if ref_rounded else 1.0) * BF16_OWN
    ex = 0.0 if extra is None else np.asarray(extra, dtype=np.float64)
    _record(what, io, own, g, r, diff, own_k, ex)
    if io == "f32":
        err = float(diff.max())
        assert err <= 1e-4, f"{what}: max abs err {err:.3e} > 1e-4"
        return
    scale = rms(r)
    rel = rms(g - r) / scale if scale > 0 else rms(g - r)
    assert rel <= BF16_REL, f"{what}: RMS err / RMS(ref) = {rel:.3e} > {BF16_REL}"
    bound = BF16_REL * scale + (own_k * np.abs(r) if own else 0.0) + ex
    worst = np.unravel_index(np.argmax(diff - bound), diff.shape)
    assert (diff <= bound).all(), (f"{what}: element {worst}: |err| {diff[worst]:.3e} > "
                                   f"{float(np.broadcast_to(bound, diff.shape)[worst]):.3e} "
                                   f"(ref {r[worst]:.3e}, RMS {scale:.3e}, stored {stored})")


def assert_attention_close(got, case_f64: dict, seqs, what: str = "attention o"):
    """The attention outputs ``got[seqs]`` against the oracle (see the module docstring): within
    the bf16 rule of the oracle on the bf16-rounded rotated query, and within that rule plus the
    oracle's own change under that rounding of the plain fp64 oracle.  Returns the plain
    oracle's (outputs, rotated node keys)."""
    from oracle import attention as A
    o_ref, kr_ref = A.tree_attention(case_f64, batch=seqs)
    o_rq, _ = A.tree_attention(case_f64, batch=seqs, query_bf16=True)
    g = got[seqs]
    assert_close(g, o_rq[seqs], "bf16", what + " (bf16 query)")
    assert_close(g, o_ref[seqs], "bf16", what, extra=np.abs(o_rq[seqs] - o_ref[seqs]))
    return o_ref, kr_ref


def margin_summary() -> list[str]:
    """Worst margins per compared quantity (labels with a trailing ' b=..' or node index merged)."""
    import re
    agg: dict = {}
    for m in MARGINS:
        if m["io"] == "f32" or "max_over_rms" not in m:
            continue
        key = (re.sub(r" (b=)?\d+$", "", m["what"]),
               ("bf16x2" if m.get("own_k", BF16_OWN) > BF16_OWN else "bf16") if m["stored_bf16"] else "f32")
        a = agg.setdefault(key, dict(calls=0, n=0, over=0, max_over_rms=0.0, rms=0.0, worst=0.0))
        a["calls"] += 1
        a["n"] += m["n"]
        a["over"] += m["n_over_strict"]
        a["max_over_rms"] = max(a["max_over_rms"], m["max_over_rms"])
        a["rms"] = max(a["rms"], m["rms_err_over_rms"])
        a["worst"] = max(a["worst"], m["worst_vs_bound"])
    lines = [f"{'bf16-I/O tensor':<46} {'stored':>6} {'calls':>5} {'max|err|/RMS':>12} {'RMS(err)/RMS':>12} "
             f"{'elems>2e-2RMS':>14} {'worst/bound':>11}"]
    for (what, st), a in agg.items():
        lines.append(f"{what:<46} {st:>6} {a['calls']:>5} {a['max_over_rms']:>12.4f} {a['rms']:>12.4f} "
                     f"{a['over']:>7}/{a['n']:<9} {a['worst']:>8.3f}")
    return lines


def _err(B: int) -> torch.Tensor:
    return torch.full((B,), 12345, dtype=torch.int32, device=DEV)


def gdn_inputs(case: W.GDNCase) -> dict:
    return dict(q=to_dev(case.q), k=to_dev(case.k), v=to_dev(case.v), alpha=to_dev(case.alpha),
                beta=to_dev(case.beta), S0=to_dev(case.S0), parents=to_dev(case.parents))


def run_tree_prepare(parents: torch.Tensor, path_cap: int | None = None) -> dict:
    """Depth and mask bits; with path_cap, also the root-to-node paths and the maximum depth."""
    B, N = parents.shape
    p = to_dev(parents)
    depth = torch.full((B, N), -7, dtype=torch.int32, device=DEV)
    bits = torch.zeros((B, N, (N + 31) // 32), dtype=torch.int32, device=DEV)
    err = _err(B)
    paths = maxd = None
    if path_cap is not None:
        paths = torch.full((B, N, path_cap), 777, dtype=torch.int32, device=DEV)
        maxd = torch.full((B,), 777, dtype=torch.int32, device=DEV)
    tv.tv_tree_prepare(p, depth, bits, err, paths=paths, max_depth=maxd)
    torch.cuda.synchronize()
    r = dict(depth=depth.cpu(), mask_bits=bits.cpu().numpy().view(np.uint32), err=err.cpu())
    if path_cap is not None:
        r.update(paths=paths.cpu().numpy(), max_depth=maxd.cpu().numpy())
    return r


def run_fork(case: W.GDNCase, inputs: dict | None = None, keep_device: bool = False) -> dict:
    x = gdn_inputs(case) if inputs is None else inputs
    B, N, H, dk, dv = case.shape
    out = torch.full((B, N, H, dv), float("nan"), dtype=x["q"].dtype, device=DEV)
    states = torch.full((B, N, H, dv, dk), float("nan"), dtype=x["S0"].dtype, device=DEV)
    err = _err(B)
    tv.tv_gdn_tree_verify_fork(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"], x["parents"], out,
                               states, err, q_scale=case.q_scale)
    torch.cuda.synchronize()
    if keep_device:
        return dict(out=out, states=states, err=err, inputs=x)
    return dict(out=out.cpu(), states=states.cpu(), err=err.cpu(), inputs=x)


def run_wy(case: W.GDNCase, inputs: dict | None = None) -> dict:
    x = gdn_inputs(case) if inputs is None else inputs
    B, N, H, dk, dv = case.shape
    out = torch.full((B, N, H, dv), float("nan"), dtype=x["q"].dtype, device=DEV)
    pv = torch.full((B, N, H, dv), float("nan"), dtype=torch.float32, device=DEV)
    lg = torch.full((B, N, H), float("nan"), dtype=torch.float32, device=DEV)
    err = _err(B)
    tv.tv_gdn_tree_verify_wy(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"], x["parents"], out, pv,
                             lg, err, q_scale=case.q_scale)
    torch.cuda.synchronize()
    return dict(out=out.cpu(), pseudo_v=pv.cpu(), log_gamma=lg.cpu(), err=err.cpu(), inputs=x,
                pv_dev=pv, lg_dev=lg)


def run_commit(case: W.GDNCase, mode: str, verify: dict, path=None, path_len=None) -> torch.Tensor:
    """Commit after a verify call (``verify`` is what run_fork / run_wy returned); returns S_0."""
    x = verify["inputs"]
    S0 = x["S0"].clone()
    B = S0.shape[0]
    err = _err(B)
    p = to_dev(case.path if path is None else path)
    L = to_dev(case.path_len if path_len is None else path_len)
    if mode == "fork":
        states = verify["states"]
        states = states if states.is_cuda else to_dev(states)
        tv.tv_gdn_commit(tv.TV_MODE_FORK, p, L, x["parents"], S0, err, node_states=states)
    else:
        tv.tv_gdn_commit(tv.TV_MODE_WY, p, L, x["parents"], S0, err, pseudo_v=verify["pv_dev"],
                         log_gamma=verify["lg_dev"], k=x["k"])
    torch.cuda.synchronize()
    verify["commit_err"] = err.cpu()
    return S0.cpu()


def f32np(t: torch.Tensor) -> np.ndarray:
    """Stored values as float32 numpy (exact for bf16): for the large paged caches."""
    return t.detach().cpu().float().numpy()


def attn_f64(case: W.AttnCase) -> dict:
    """Oracle inputs: q / k / v in fp64; the paged caches as exact float32 (the oracle upcasts
    the rows it gathers)."""
    return dict(q=W.f64(case.q), k_new=W.f64(case.k_new), v_new=W.f64(case.v_new),
                k_cache=f32np(case.k_cache), v_cache=f32np(case.v_cache),
                block_table=case.block_table.numpy(), prefix_len=case.prefix_len.numpy(),
                parents=case.parents.numpy(), rope_theta=case.rope_theta)


def run_attn(case: W.AttnCase, keep_device: bool = False) -> dict:
    B, N, Hq, Hkv, hd = case.shape
    q, kn, vn = to_dev(case.q), to_dev(case.k_new), to_dev(case.v_new)
    kc, vc = to_dev(case.k_cache), to_dev(case.v_cache)
    table, plen, par = to_dev(case.block_table), to_dev(case.prefix_len), to_dev(case.parents)
    out = torch.full((B, N, Hq, hd), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws_bytes = tv.tv_tree_attn_workspace_size(B, N, Hq, Hkv, hd, table.shape[1])
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    err = _err(B)
    tv.tv_tree_attn(q, kn, vn, kc, vc, table, plen, par, out, ws, err, rope_theta=case.rope_theta)
    torch.cuda.synchronize()
    if keep_device:
        return dict(out=out, k_cache=kc, v_cache=vc, err=err)
    return dict(out=out.cpu(), k_cache=kc.cpu(), v_cache=vc.cpu(), err=err.cpu())


def run_compact(case: W.AttnCase, k_cache: torch.Tensor, v_cache: torch.Tensor, path=None,
                path_len=None) -> dict:
    B = case.q.shape[0]
    kc, vc = to_dev(k_cache), to_dev(v_cache)
    p = to_dev(case.path if path is None else path)
    L = to_dev(case.path_len if path_len is None else path_len)
    slot_map = torch.full(p.shape, 777, dtype=torch.int32, device=DEV)
    new_len = torch.full((B,), 777, dtype=torch.int32, device=DEV)
    err = _err(B)
    tv.tv_kv_compact(kc, vc, to_dev(case.block_table), to_dev(case.prefix_len), to_dev(case.parents), p, L,
                     slot_map, new_len, err)
    torch.cuda.synchronize()
    return dict(k_cache=kc.cpu(), v_cache=vc.cpu(), slot_map=slot_map.cpu().numpy(),
                new_len=new_len.cpu().numpy(), err=err.cpu())


def run_compact_remap(k_cache, v_cache, block_table, prefix_len, parents, path, path_len,
                      table_out_fill: int = -7) -> dict:
    """``tv_kv_compact_remap`` on device copies of the given tensors.  The caches stay on the
    device (the full-size tests gather rows from them); the small outputs come back as numpy."""
    B = block_table.shape[0]
    kc, vc = to_dev(k_cache), to_dev(v_cache)
    table = to_dev(block_table)
    table_out = torch.full_like(table, table_out_fill)
    p = to_dev(path)
    slot_map = torch.full(p.shape, 777, dtype=torch.int32, device=DEV)
    new_len = torch.full((B,), 777, dtype=torch.int32, device=DEV)
    remapped = torch.full((B,), 777, dtype=torch.int32, device=DEV)
    err = _err(B)
    tv.tv_kv_compact_remap(kc, vc, table, table_out, to_dev(prefix_len), to_dev(parents), p, to_dev(path_len),
                           slot_map, new_len, remapped, err)
    torch.cuda.synchronize()
    return dict(k_cache=kc, v_cache=vc, table=table_out.cpu().numpy(), slot_map=slot_map.cpu().numpy(),
                new_len=new_len.cpu().numpy(), remapped=remapped.cpu().numpy(), err=err.cpu())
