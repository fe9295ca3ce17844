"""Helpers for the GPU tests: move a workload to the device, run the library
through its C ABI binding, and compare with the oracle."""
import dataclasses

import numpy as np
import torch

import fd_synth as syn

# Tolerances (the stated bounds: max-abs error <= 1e-2 and max-rel error
# <= 1e-2 on O, 1e-3 absolute on LSE).  O passes elementwise when
# |o - r| <= ATOL + RTOL |r|, and in addition the relative error over the
# elements with |r| >= REL_FLOOR must stay within O_MAX_REL: a relative
# error is meaningless next to zero, and O entries are weighted means of
# N(0,1) values, so many sit near it.
O_ATOL, O_RTOL, LSE_ATOL = 1e-2, 1e-2, 1e-3
O_MAX_REL, REL_FLOOR = 1e-2, 1e-2


def dev_bf16(bits, device="cuda", dtype="bf16"):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16)


def dev_fp8(codes, device="cuda"):
    """FP8 codes as a uint8 CUDA tensor (the binding takes kv_dtype with it)."""
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).to(device)


def to_device(w, device="cuda"):
    dt = getattr(w, "dtype", "bf16")
    if getattr(w, "kv_dtype", None) in ("e4m3", "e5m2"):
        k, v = dev_fp8(w.k, device), dev_fp8(w.v, device)
    else:
        k, v = dev_bf16(w.k, device, dt), dev_bf16(w.v, device, dt)
    d = dict(q=dev_bf16(w.q, device, dt), k=k, v=v,
             seq_lens=torch.from_numpy(np.ascontiguousarray(w.seq_lens, dtype=np.int32)).to(device))
    if w.paged:
        d["block_table"] = torch.from_numpy(np.ascontiguousarray(w.block_table, dtype=np.int32)).to(device)
    return d


def run(w, dev=None, **kw):
    """Run fd_decode / fd_decode_paged on workload w; returns fp64 numpy (O, LSE)."""
    import decode_attention_decoding_gb300 as fd
    dev = dev or to_device(w)
    if getattr(w, "kv_dtype", None) in ("e4m3", "e5m2"):
        kw = dict(kw, kv_dtype=w.kv_dtype, k_scale=w.k_scale, v_scale=w.v_scale)
    if w.paged:
        o, l = fd.fd_decode_paged(dev["q"], dev["k"], dev["v"], dev["block_table"], dev["seq_lens"],
                                  seq_lens_host=torch.from_numpy(w.seq_lens), scale=w.scale, **kw)
    else:
        o, l = fd.fd_decode(dev["q"], dev["k"], dev["v"], dev["seq_lens"],
                            seq_lens_host=torch.from_numpy(w.seq_lens), scale=w.scale, **kw)
    torch.cuda.synchronize()
    return o.cpu().numpy().astype(np.float64), (None if l is None else l.cpu().numpy().astype(np.float64))


def check(o, lse, ro, rl, what=""):
    """Assert the tolerances; return (max_abs_O, max_rel_O over |r|>=1e-2, max_abs_LSE)."""
    err = np.abs(o - ro)
    bad = err > O_ATOL + O_RTOL * np.abs(ro)
    assert not bad.any(), f"{what}: {int(bad.sum())} O elements out of tolerance, max err {err.max():.3g}"
    big = np.abs(ro) >= REL_FLOOR
    max_rel = float((err[big] / np.abs(ro[big])).max()) if big.any() else 0.0
    assert max_rel <= O_MAX_REL, f"{what}: max relative O error {max_rel:.3g} over |r| >= {REL_FLOOR}"
    lse_err = 0.0
    if lse is not None:
        fin = np.isfinite(rl)
        assert np.array_equal(fin, np.isfinite(lse)), f"{what}: LSE finiteness differs"
        assert np.all(lse[~fin] == rl[~fin]), f"{what}: infinite LSE differs"
        if fin.any():
            lse_err = float(np.abs(lse[fin] - rl[fin]).max())
            assert lse_err <= LSE_ATOL, f"{what}: LSE err {lse_err:.3g}"
    return float(err.max()) if err.size else 0.0, max_rel, lse_err


def contig_to_paged(w, page, perm_seed, extra_pages=3, poison=False):
    """Same logical K/V in shuffled pages (unreferenced slots NaN when poison)."""
    B, S, hkv, d = w.k.shape
    lens = w.seq_lens
    used = sum((int(L) + page - 1) // page for L in lens)
    n_pages = used + extra_pages
    perm = syn.permutation(perm_seed, n_pages)
    max_blocks = max(1, (S + page - 1) // page)
    table = syn.build_block_table(lens, page, max_blocks, perm)
    fp8 = getattr(w, "kv_dtype", None) in ("e4m3", "e5m2")
    nan = np.uint8(0x7F) if fp8 else syn.BF16_NAN          # a NaN code in both FP8 formats
    fill = nan if poison else w.k.dtype.type(0)
    kp = np.full((n_pages, page, hkv, d), fill, w.k.dtype)
    vp = np.full((n_pages, page, hkv, d), fill, w.v.dtype)
    for b in range(B):
        L = int(lens[b])
        nb = (L + page - 1) // page
        for i in range(nb):
            n = min(page, L - i * page)
            kp[table[b, i], :n] = w.k[b, i * page:i * page + n]
            vp[table[b, i], :n] = w.v[b, i * page:i * page + n]
    return dataclasses.replace(w, name=w.name + f"_p{page}", k=kp, v=vp, seq_lens=lens.copy(),
                               page_size=page, block_table=table)


def sample_items(w, n, seed=0):
    """A spread of (b, h) query rows: first/last request and head, plus random ones."""
    rng = np.random.default_rng(seed)
    B, hq = w.batch, w.num_q_heads
    pairs = {(0, 0), (B - 1, hq - 1), (0, hq - 1), (B - 1, 0)}
    while len(pairs) < min(n, B * hq):
        pairs.add((int(rng.integers(B)), int(rng.integers(hq))))
    return np.array([[b, h, 0, -1] for b, h in sorted(pairs)], dtype=np.int32)


def small_page_twin_flags(w):
    """Flags that make a contiguous run of w take the consumers that a paged
    run with pages under 8 tokens takes, so the two agree bitwise: the
    unfused tensor-core consumers when a kv head has 2 or more query columns
    (G x q_len) and a row holds at least 128 bytes, else CUDA cores."""
    cols = (w.num_q_heads // w.num_kv_heads) * w.q_len
    row_bytes = w.head_dim * w.kv_elem_bytes
    return 0x8 if cols >= 2 and row_bytes >= 128 else 0x2   # FD_FLAG_NO_HEAD_FUSION / FD_FLAG_CUDA_CORES


repage = syn.repage   # the same logical K/V in shuffled pages of another size
