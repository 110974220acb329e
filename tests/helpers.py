"""Shared helpers of the GPU parity tests."""
import numpy as np

ATOL, RTOL = 1e-2, 2e-2   # |gpu - ref| <= ATOL + RTOL * |ref| per element (out and lse)


def np64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(gpu, ref, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    both_inf = np.isneginf(gpu) & np.isneginf(ref)
    g = np.where(both_inf, 0.0, gpu)
    r = np.where(both_inf, 0.0, ref)
    err = np.abs(g - r)
    bad = ~(err <= ATOL + RTOL * np.abs(r))
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; first at "
                             f"{tuple(i)}: gpu={gpu[tuple(i)]} ref={ref[tuple(i)]}; max abs err {err.max():.3e}")
    return float(err.max()) if err.size else 0.0


def workload_arrays(wl):
    """Oracle inputs: the bf16 values of the workload as fp64 numpy arrays."""
    return dict(q=np64(wl.q), k_chunk=np64(wl.k_chunk), v_chunk=np64(wl.v_chunk),
                k_pool=np64(wl.k_pool), v_pool=np64(wl.v_pool))


def empty_sequence_specs():
    """Prefill sequences with nothing to recompute between sequences that have chunk rows."""
    from segmented_kv_attention_msa_b300 import workload as W
    return [W.SeqSpec([(0, 64)], np.arange(64, 100)), W.SeqSpec([(0, 48)], np.array([], np.int64)),
            W.SeqSpec([], np.arange(0, 20)), W.SeqSpec([(16, 32)], np.array([], np.int64))]


class DevicePool:
    """The oracle's view of a device pool tensor [blocks][Hkv][16][d]: indexing by (block
    ids, :, slots, :) copies just those rows to the host as fp64.  The oracle gathers each
    sequence's keys by block and slot; turning a multi-GB pool into fp64 on the host first
    would take tens of GB of host memory.  Only data movement happens here."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, idx):
        import torch
        b, _, s, _ = idx
        bi = torch.as_tensor(np.asarray(b), dtype=torch.long, device=self.t.device)
        si = torch.as_tensor(np.asarray(s), dtype=torch.long, device=self.t.device)
        return np64(self.t[bi, :, si, :])


def export_tables(plan_export):
    """Split a canonical plan export into its tables (tokens, KV tiles, query tiles, classes)."""
    e = np.asarray(plan_export, np.int64)
    mode, nseq, ntok, nkt, nqt, ncls = (int(x) for x in e[:6])
    o = 6
    tok = e[o:o + 4 * ntok].reshape(-1, 4)
    o += 4 * ntok
    kt = e[o:o + 6 * nkt].reshape(-1, 6)
    o += 6 * nkt
    qt = e[o:o + 5 * nqt].reshape(-1, 5)
    o += 5 * nqt
    cls = e[o:o + ncls]
    return tok, kt, qt, cls
