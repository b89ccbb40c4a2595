"""Device-resident ternary decoder for ``decode_step_t158``.

Holds the model's device tensors (torch provides the memory), fills the
``t158_model`` descriptor, and owns the KV cache and the workspace.  All
arithmetic happens in libqlin: weights are packed by ``t158_pack`` (host C),
RoPE tables by ``t158_rope_table`` (GPU), and every forward step by
``decode_step_t158``.
"""
from __future__ import annotations

import numpy as np
import torch

from . import qlin

MATRIX_ORDER = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


class T158Decoder:
    def __init__(self, cfg, weights, device="cuda"):
        """cfg: object with n_layers, dim, n_heads, n_kv_heads, head_dim, ffn, vocab, max_pos, eps,
        rope_base and matrices() -> [(name, rows, cols)]; weights: dict of numpy arrays with
        per-layer int8 trit matrices, scales [L][7], g_attn/g_ffn [L][dim], g_final [dim],
        emb bf16 bits [vocab][dim]."""
        self.cfg = cfg
        dev = torch.device(device)
        L = cfg.n_layers
        dims = {name: (n, k) for name, n, k in cfg.matrices()}
        self.w = []
        self.pitch = []
        for name in MATRIX_ORDER:
            n, k = dims[name]
            pitch = qlin.t158_pitch(k)
            host = np.empty((L, n, pitch), np.uint8)
            for l in range(L):
                host[l] = qlin.t158_pack(weights["layers"][l][name], pitch)
            self.w.append(torch.from_numpy(host).to(dev))
            self.pitch.append(pitch)
        f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
        self.scales = f32(weights["scales"])
        self.g_attn = f32(weights["g_attn"])
        self.g_ffn = f32(weights["g_ffn"])
        self.g_final = f32(weights["g_final"])
        self.emb = torch.from_numpy(np.ascontiguousarray(weights["emb"]).view(np.int16)).to(dev)
        half = cfg.head_dim // 2
        self.rope_cos = torch.empty((cfg.max_pos, half), dtype=torch.float32, device=dev)
        self.rope_sin = torch.empty((cfg.max_pos, half), dtype=torch.float32, device=dev)
        qlin.t158_rope_table(self.rope_cos, self.rope_sin, cfg.max_pos, cfg.head_dim, cfg.rope_base)

        m = qlin.T158ModelC()
        m.n_layers, m.dim, m.n_heads, m.n_kv_heads = L, cfg.dim, cfg.n_heads, cfg.n_kv_heads
        m.head_dim, m.ffn, m.vocab, m.max_pos = cfg.head_dim, cfg.ffn, cfg.vocab, cfg.max_pos
        m.eps = cfg.eps
        for j in range(len(MATRIX_ORDER)):
            m.w[j] = self.w[j].data_ptr()
            m.pitch[j] = self.pitch[j]
        m.scales, m.g_attn, m.g_ffn = self.scales.data_ptr(), self.g_attn.data_ptr(), self.g_ffn.data_ptr()
        m.g_final, m.emb = self.g_final.data_ptr(), self.emb.data_ptr()
        m.rope_cos, m.rope_sin = self.rope_cos.data_ptr(), self.rope_sin.data_ptr()
        self.model = m
        self.ws_bytes = qlin.decode_step_t158_workspace_size(m)
        self.workspace = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.kv = torch.zeros((L, 2, cfg.max_pos, cfg.kv_dim), dtype=torch.float32, device=dev)
        self.token = torch.zeros(1, dtype=torch.int32, device=dev)
        self.logits = torch.empty(cfg.vocab, dtype=torch.float32, device=dev)

    def weight_bytes(self) -> int:
        """Packed bytes at the canonical ceil(K/5) pitch, as the roofline counts them."""
        total = 0
        for name, n, k in self.cfg.matrices():
            total += self.cfg.n_layers * n * ((k + 4) // 5)
        return total

    def step(self, pos: int, token=None, logits: bool = True, stream=None):
        """One forward step at `pos` for the token in self.token (or `token`, a device int32 tensor);
        the greedy token is written back to self.token (so steps chain on the device)."""
        tok = self.token if token is None else token
        qlin.decode_step_t158(self.model, self.kv, self.workspace, self.ws_bytes, tok, pos,
                              self.logits if logits else None, self.token, stream)

    def check_status(self, stream=None):
        qlin.decode_step_t158_status(self.workspace, stream)

    # ---------------------------------------------------------------- sketch head
    def prepare_sketch(self, k: int = 32, n_cand: int = 1024, stream=None):
        """Tables of the sketch head over the tied table, ordered by the final norm gain,
        and the workspace of ``step_sketch``."""
        cfg, dev = self.cfg, self.emb.device
        self.sk_emb_t = torch.empty((cfg.dim, qlin.qlin_sketch_emb_t_pitch(cfg.vocab)), dtype=torch.int16,
                                    device=dev)
        self.sk_signs = torch.empty(qlin.qlin_sketch_signs_bytes(cfg.vocab, cfg.dim) // 8, dtype=torch.int64,
                                    device=dev)
        self.sk_perm = torch.empty(cfg.dim, dtype=torch.int32, device=dev)
        self.sk_ce = torch.zeros(1, dtype=torch.float32, device=dev)
        qlin.qlin_sketch_prepare(self.emb, cfg.vocab, cfg.dim, self.g_final, self.sk_emb_t, self.sk_signs,
                                 self.sk_perm, self.sk_ce, stream)
        sk = qlin.T158SketchC()
        sk.emb_t, sk.signs = self.sk_emb_t.data_ptr(), self.sk_signs.data_ptr()
        sk.perm, sk.c_e = self.sk_perm.data_ptr(), self.sk_ce.data_ptr()
        sk.k, sk.n_cand = k, n_cand
        self.sketch = sk
        self.sk_ws_bytes = qlin.decode_step_t158_sketch_workspace_size(self.model, sk)
        self.sk_workspace = torch.zeros(self.sk_ws_bytes, dtype=torch.uint8, device=dev)

    def step_sketch(self, pos: int, token=None, stream=None):
        """One forward step whose next token comes from the sketch head (two launches)."""
        tok = self.token if token is None else token
        qlin.decode_step_t158_sketch(self.model, self.sketch, self.kv, self.sk_workspace, self.sk_ws_bytes, tok, pos,
                                     self.token, stream)

    def check_sketch_status(self, stream=None):
        qlin.decode_step_t158_sketch_status(self.model, self.sketch, self.sk_workspace, stream)

    # ---------------------------------------------------------------- lanes
    def prepare_lanes(self, n_seqs: int, max_lanes: int):
        """KV caches for n_seqs sequences and the workspace of ``step_lanes``."""
        cfg, dev = self.cfg, self.emb.device
        self.n_seqs, self.max_lanes = n_seqs, max_lanes
        self.kv_lanes = torch.zeros((n_seqs, cfg.n_layers, 2, cfg.max_pos, cfg.kv_dim), dtype=torch.float32,
                                    device=dev)
        self.lanes_ws_bytes = qlin.decode_lanes_t158_workspace_size(self.model, max_lanes)
        self.lanes_workspace = torch.zeros(self.lanes_ws_bytes, dtype=torch.uint8, device=dev)
        self.lane_tokens = torch.zeros(max_lanes, dtype=torch.int32, device=dev)
        self.lane_pos = torch.zeros(max_lanes, dtype=torch.int32, device=dev)
        self.lane_seq = torch.zeros(max_lanes, dtype=torch.int32, device=dev)
        self.lane_next = torch.zeros(max_lanes, dtype=torch.int32, device=dev)

    def step_lanes(self, n_lanes: int, logits=None, stream=None):
        """One step over lanes 0..n_lanes-1 of lane_tokens / lane_pos / lane_seq; the greedy tokens go to
        lane_next (and the logits [n_lanes][vocab] to ``logits`` if given)."""
        qlin.decode_lanes_t158(self.model, self.kv_lanes, self.n_seqs, n_lanes, self.lane_tokens, self.lane_pos,
                               self.lane_seq, logits, self.lane_next, self.lanes_workspace, self.lanes_ws_bytes,
                               self.max_lanes, stream)

    def check_lanes_status(self, stream=None):
        qlin.decode_lanes_t158_status(self.lanes_workspace, stream)
