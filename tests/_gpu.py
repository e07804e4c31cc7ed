"""GPU runners for the parity tests: each runs one C-ABI call through the binding on the
seeded inputs of a ``workloads`` case and returns the outputs as CPU tensors.  Plus the
tolerance rule shared by the tests.

Tolerance of the floating-point outputs:
  * fp32 I/O: max |x - ref| <= 1e-4.
  * bf16 I/O with fp32 arithmetic, "within 2e-2 relative to the per-tensor RMS", read as two
    conditions over the compared tensor:
      RMS(x - ref) <= 2e-2 * RMS(ref)                         (the stated bound), and
      |x - ref| <= 2e-2 * RMS(ref) + 2^-7 * |ref| per element  (no outlier; the second term
                                                              is four bf16 roundings of the
                                                              element's own magnitude, the
                                                              least a bf16 result can carry).
Integer outputs are compared exactly.
"""
from __future__ import annotations

import numpy as np
import torch

import tree_speculative_verification_gdn_gb300 as tv
import workloads as W

DEV = "cuda"


def to_dev(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().to(DEV)


BF16_REL = 2e-2
BF16_OWN = 2.0 ** -7


def rms(x: np.ndarray) -> float:
    x = np.asarray(x, dtype=np.float64)
    return float(np.sqrt(np.mean(x * x))) if x.size else 0.0


def max_err(got, ref) -> float:
    g = W.f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    return float(np.abs(g - np.asarray(ref, dtype=np.float64)).max())


def assert_close(got, ref, io: str, what: str) -> None:
    g = W.f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, f"{what}: shape {g.shape} vs {r.shape}"
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    if not g.size:
        return
    diff = np.abs(g - r)
    if io == "f32":
        err = float(diff.max())
        assert err <= 1e-4, f"{what}: max abs err {err:.3e} > 1e-4"
        return
    scale = rms(r)
    rel = rms(g - r) / scale if scale > 0 else rms(g - r)
    assert rel <= BF16_REL, f"{what}: RMS err / RMS(ref) = {rel:.3e} > {BF16_REL}"
    bound = BF16_REL * scale + BF16_OWN * np.abs(r)
    worst = np.unravel_index(np.argmax(diff - bound), diff.shape)
    assert (diff <= bound).all(), (f"{what}: element {worst}: |err| {diff[worst]:.3e} > "
                                   f"{bound[worst]:.3e} (ref {r[worst]:.3e}, RMS {scale:.3e})")


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
