"""Helpers shared by the GPU tests: seeded inputs placed on the device, oracle runs, parity metrics.

The oracle and the CUDA library see the same seeded inputs (from synth); expected values come
only from the oracle.
"""
from __future__ import annotations

import numpy as np

import synth

INDEX_GAP = 1e-5   # near-tie rule for top-k indices (oracle 16th vs 17th logit)
# Gates, matched by expert id: the tensor-core router's logits carry ~1e-5 of the MMA's accumulation
# rounding where they are not recomputed (every expert whose place could depend on it is), which moves
# a gate by up to ~1.5e-5; the CUDA-core router's fp32 dot products give ~1e-6.
GATE_TOL = 5e-5
REL_TOL = 2e-3     # max|y_gpu - y_ref| / max|y_ref|


def _image(tile: np.ndarray) -> np.ndarray:
    """Scale image of one 128-row tile ([..., 128, nb] bytes): row 32c + i, block 4g + e -> 512g + 16i + 4c + e."""
    lead, nb = tile.shape[:-2], tile.shape[-1]
    t = tile.reshape(*lead, 4, 32, nb // 4, 4)                      # [c][i][g][e]
    k = len(lead)
    return t.transpose(*range(k), k + 2, k + 1, k, k + 3).reshape(*lead, 128 * nb)  # [g][i][c][e]


def device_order(records: np.ndarray, d: int, f: int) -> np.ndarray:
    """Host restatement of the device order (include/k3moe.h, k3moe_pack_records) for records in the
    stored order, one per row of `records`. Gate/up: stacked tile 2u + h (rows 0-63: gate rows
    128u + 64h.., rows 64-127: up rows 128u + 64h..) replaces gate tile u (h = 0) or up tile u (h = 1),
    codes and scales; down: each tile's scales. Every tile's scales are stored as its image."""
    out = records.copy()
    n = len(records)
    nc, ns = d * f // 2, d * f // 32
    u = f // 128
    g_c, u_c = slice(0, nc), slice(nc + ns, 2 * nc + ns)
    g_s, u_s = slice(nc, nc + ns), slice(2 * nc + ns, 2 * (nc + ns))
    gc = records[:, g_c].reshape(n, u, 2, 64, d // 2)   # [tile][half][row][bytes]
    uc = records[:, u_c].reshape(n, u, 2, 64, d // 2)
    out[:, g_c] = np.stack([gc[:, :, 0], uc[:, :, 0]], axis=2).reshape(n, nc)   # stacked tiles 2u
    out[:, u_c] = np.stack([gc[:, :, 1], uc[:, :, 1]], axis=2).reshape(n, nc)   # stacked tiles 2u + 1
    gs = records[:, g_s].reshape(n, u, 2, 64, d // 32)
    us = records[:, u_s].reshape(n, u, 2, 64, d // 32)
    out[:, g_s] = _image(np.concatenate([gs[:, :, 0], us[:, :, 0]], axis=2)).reshape(n, ns)
    out[:, u_s] = _image(np.concatenate([gs[:, :, 1], us[:, :, 1]], axis=2)).reshape(n, ns)
    off = 2 * (nc + ns) + nc
    ds = records[:, off:off + ns].reshape(n, d // 128, 128, f // 32)
    out[:, off:off + ns] = _image(ds).reshape(n, ns)
    return out


class DeviceLayer:
    """One layer's inputs on the GPU (records generated on the device, then put in the device scale
    order unless pack=False) plus the host copies (stored order) the oracle needs."""

    def __init__(self, shape: synth.LayerShape, seed: int, layer: int = 0, zipf_s: float | None = None,
                 x_dtype: str = "bf16", stride: int | None = None, pack: bool = True, score: str = "softmax",
                 shared_format: str = "mxfp4", act: str = "exact"):
        import torch
        import mxfp4_routed_expert_k3moe_gb300 as k3
        self.shape, self.seed, self.layer, self.x_dtype, self.score = shape, seed, layer, x_dtype, score
        self.shared_format = shared_format
        self.stride = stride or shape.record_stride
        E, S = shape.n_routed, shape.n_shared
        self.W_host = synth.router_weights(shape, seed, layer)
        self.bias_host = None if zipf_s is None else synth.zipf_bias(shape, seed, zipf_s, layer)
        dev = torch.device("cuda")
        self.W = torch.from_numpy(self.W_host).to(dev)
        self.bias = None if self.bias_host is None else torch.from_numpy(self.bias_host).to(dev)
        self.routed = torch.empty(E * self.stride, dtype=torch.uint8, device=dev)
        self.shared = torch.empty(max(1, S) * self.stride, dtype=torch.uint8, device=dev)
        st = torch.cuda.current_stream().cuda_stream
        synth.records_device(shape, seed, layer, 0, E, self.routed.data_ptr(), self.stride, st)
        self.sstride = 0
        if S and shared_format == "bf16":  # bf16 shared records, drawn on the host, used as stored
            self.sstride = synth.shared_bf16_stride(shape)
            self.set_shared_bf16(synth.shared_records_bf16(shape, seed, layer, S, self.sstride))
        elif S:
            synth.records_device(shape, seed, layer, E, S, self.shared.data_ptr(), self.stride, st)
        self.cfg = k3.Config.make(shape.d_model, shape.d_ff, E, shape.top_k, S,
                                  x_dtype=k3.X_BF16 if x_dtype == "bf16" else k3.X_F32, record_stride=self.stride,
                                  score_func=k3.SCORE_SOFTMAX if score == "softmax" else k3.SCORE_SIGMOID_BIAS,
                                  record_order=k3.ORDER_DEVICE if pack else k3.ORDER_STORED,
                                  shared_format=k3.SHARED_BF16 if shared_format == "bf16" else k3.SHARED_MXFP4,
                                  shared_stride=self.sstride,
                                  act_mode=k3.ACT_BF16H if act == "bf16h" else k3.ACT_EXACT)
        if pack:
            k3.pack_records(self.cfg, self.routed, E)
            if S and shared_format == "mxfp4":
                k3.pack_records(self.cfg, self.shared, S)
        self._host_records = {}

    def set_shared_bf16(self, recs: np.ndarray):
        """bf16 shared records (uint16 [S, sstride / 2]) on the device and for the oracle."""
        import torch
        self.shared_bf16_host = np.ascontiguousarray(recs, dtype=np.uint16)
        self.shared = torch.from_numpy(self.shared_bf16_host.view(np.uint8).reshape(-1).copy()).cuda()

    def shared_host(self):
        """The shared records the oracle takes (MXFP4 records, or bf16 ones)."""
        sh = self.shape
        if self.shared_format == "bf16":
            return [r for r in self.shared_bf16_host]
        return list(self.host_records([sh.n_routed + s for s in range(sh.n_shared)]).values())

    def host_records(self, experts):
        need = [e for e in experts if e not in self._host_records]
        if need:
            recs = synth.records_host(self.shape, self.seed, self.layer, need, self.stride)
            for e, r in zip(need, recs):
                self._host_records[e] = r
        return {e: self._host_records[e] for e in experts}

    def tokens(self, T: int, batch: int = 0):
        """(host array, device tensor) of T seeded tokens."""
        import torch
        xh = synth.tokens(self.shape, self.seed, T, self.x_dtype, batch)
        xd = torch.from_numpy(xh.view(np.int16) if self.x_dtype == "bf16" else xh).cuda()
        return xh, xd

    def oracle(self, xh: np.ndarray, token_ids=None):
        """Oracle y, idx, w, logits for the given host tokens (optionally a subset of rows)."""
        import oracle
        sh = self.shape
        x = xh if token_ids is None else xh[np.asarray(token_ids)]
        xf = synth.tokens_as_f64(x, self.x_dtype)
        # route first (cheap) to know which records the oracle needs
        experts = set()
        for t in range(x.shape[0]):
            _, idx, _ = oracle.route_token(xf[t], self.W_host, sh.top_k, self.bias_host, score=self.score)
            experts.update(int(e) for e in idx)
        routed = self.host_records(sorted(experts))
        return oracle.layer(x, self.x_dtype, self.W_host, self.bias_host, routed, self.shared_host(), sh.d_model,
                            sh.d_ff, sh.top_k, score=self.score, shared_format=self.shared_format)

    def oracle_route(self, xh: np.ndarray):
        """Oracle routing of every token (logits[T, E], idx[T, k], w[T, k]), tokens in parallel."""
        import oracle
        return oracle.route_tokens(xh, self.x_dtype, self.W_host, self.shape.top_k, self.bias_host, score=self.score)

    def sel_keys(self, logits_ref: np.ndarray) -> np.ndarray:
        """The values the oracle ranked (for the near-tie rule): the logits (bias included) for the
        softmax score; sigmoid(logit) + bias for the sigmoid score."""
        if self.score == "softmax":
            return logits_ref
        from scipy.special import expit
        return expit(logits_ref) + (0.0 if self.bias_host is None else self.bias_host.astype(np.float64))

    def oracle_ffn(self, xh: np.ndarray, idx: np.ndarray, w: np.ndarray):
        """Oracle of the FFN + combine for GIVEN routing (per token: sum_i w_i o_i + sum_s o_s)."""
        import oracle
        sh = self.shape
        xf = synth.tokens_as_f64(xh, self.x_dtype)
        recs = self.host_records(sorted(set(int(e) for e in np.unique(idx))))
        shared = self.shared_host()
        run_shared = oracle.expert_token_bf16 if self.shared_format == "bf16" else oracle.expert_token
        y = np.zeros((xh.shape[0], sh.d_model))
        for t in range(xh.shape[0]):
            for e, g in zip(idx[t], w[t]):
                y[t] += float(g) * oracle.expert_token(recs[int(e)], xf[t], sh.d_model, sh.d_ff)[0]
            for r in shared:
                y[t] += run_shared(r, xf[t], sh.d_model, sh.d_ff)[0]
        return y


def oracle_order(keys: np.ndarray) -> np.ndarray:
    """The oracle's ranking of one token's experts: larger value first, equal values lower index first."""
    return np.lexsort((np.arange(len(keys)), -keys))


def index_parity(idx_gpu: np.ndarray, idx_ref: np.ndarray, keys_ref: np.ndarray, k: int):
    """The contract on the top-k indices, per token (keys_ref: the values the oracle ranked, fp64):
    * the GPU's k ids are distinct and in range;
    * the set equals the oracle's, except that where the oracle's k-th and (k+1)-th values differ by
      less than INDEX_GAP (and are not equal) the GPU may hold the (k+1)-th expert in place of the k-th:
      that exchange and no other;
    * the order: any two GPU positions i < j rank as the oracle ranks them (larger value first, equal
      values lower id first), except two experts whose values differ by less than INDEX_GAP without
      being equal. Exactly equal values get no excuse: the lower id comes first.
    Returns (ok_all, list of tokens that took the exchange, first failure message or None)."""
    near = []
    E = keys_ref.shape[1]
    for t in range(idx_ref.shape[0]):
        keys = keys_ref[t]
        g = [int(e) for e in idx_gpu[t]]
        order = oracle_order(keys)
        if [int(e) for e in order[:k]] != [int(e) for e in idx_ref[t]]:
            return False, near, f"token {t}: oracle selection is not its own ranking"
        if len(set(g)) != k or min(g) < 0 or max(g) >= E:
            return False, near, f"token {t}: GPU ids {g} not {k} distinct ids in [0, {E})"
        sg, sr = set(g), set(int(e) for e in idx_ref[t])
        if sg != sr:
            kth, k1th = int(order[k - 1]), int(order[k]) if E > k else -1
            gap = keys[kth] - keys[k1th] if k1th >= 0 else np.inf
            if not (sg - sr == {k1th} and sr - sg == {kth} and 0.0 < gap < INDEX_GAP):
                return False, near, f"token {t}: sets differ by {sorted(sg - sr)} / {sorted(sr - sg)} (gap {gap:.3g})"
            near.append(t)
        for i in range(k):
            for j in range(i + 1, k):
                a, b = g[i], g[j]
                if keys[a] > keys[b] or (keys[a] == keys[b] and a < b):
                    continue
                if keys[a] != keys[b] and abs(keys[a] - keys[b]) < INDEX_GAP:
                    continue
                return False, near, f"token {t}: positions {i}, {j} hold {a}, {b} out of the oracle's order"
    return True, near, None


def rel_err(y_gpu: np.ndarray, y_ref: np.ndarray) -> float:
    den = np.abs(y_ref).max()
    return float(np.abs(y_gpu - y_ref).max() / (den if den > 0 else 1.0))


def gate_err(idx_gpu, w_gpu, idx_ref, w_ref) -> float:
    """max |w_gpu - w_ref| over experts present in both selections (matched by expert id)."""
    err = 0.0
    for t in range(idx_ref.shape[0]):
        ref = {int(e): float(v) for e, v in zip(idx_ref[t], w_ref[t])}
        for e, v in zip(idx_gpu[t], w_gpu[t]):
            if int(e) in ref:
                err = max(err, abs(float(v) - ref[int(e)]))
    return err
