"""Shared helpers of the GPU parity tests: device transfers, layout maps between the
library's KV cache and the oracle's, and the float tolerance of the hot path."""
import numpy as np
import torch

REL_TOL = 2e-2      # max |err| <= REL_TOL * max |ref| + ABS_TOL  (layer and kernel outputs)
ABS_TOL = 1e-3


def lib():
    import __graft_entry__ as g
    g.build()
    from bit_compressed_throughput_gb300 import fg
    return fg


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.to(dtype)


def host(t):
    return t.detach().cpu().numpy()


def f16(t):
    return host(t.float()).astype(np.float64)


def assert_close(got, want, what="", rel=REL_TOL, abs_=ABS_TOL):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want).max() if got.size else 0.0
    tol = rel * (np.abs(want).max() if want.size else 0.0) + abs_
    assert err <= tol, f"{what}: max|err| {err:.4g} > tol {tol:.4g}"
    return err, tol


def cache_codes_to_rows(codes_bhtc):
    """[B][H][T][d/2] -> [B][T][h/2] (per position, heads concatenated)."""
    B, H, T, c = codes_bhtc.shape
    return codes_bhtc.transpose(0, 2, 1, 3).reshape(B, T, H * c)


def rows_to_cache(rows_btc, H):
    """[B][T][h'] -> [B][H][T][h'/H]."""
    B, T, c = rows_btc.shape
    return np.ascontiguousarray(rows_btc.reshape(B, T, H, c // H).transpose(0, 2, 1, 3))
