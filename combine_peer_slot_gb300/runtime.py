"""Device-side plumbing around the C ABI: torch allocates the inputs and
weights and provides the stream; every step of the FFN path runs in the
library's kernels (combine_peer_slot_gb300/afd.py)."""
import numpy as np

from . import afd as A
from . import workloads as W


class DeviceBytes:
    """Zero-copy uint8 view of a device allocation owned by the library, for
    inspecting or editing slot bytes from torch."""

    def __init__(self, ptr, nbytes):
        self.__cuda_array_interface__ = {"shape": (int(nbytes),), "typestr": "|u1",
                                         "data": (int(ptr), False), "version": 2}


def device_view(ptr, nbytes):
    import torch
    return torch.as_tensor(DeviceBytes(ptr, nbytes), device="cuda")


def act_tensor(a, act, device):
    """numpy activation storage (uint16 bf16 bits / float32) -> torch tensor."""
    import torch
    if act == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


class Runner:
    """One library context bound to a workload: inputs on the device, the
    layer weights registered, and helpers for pack / forward / unpack."""

    def __init__(self, w: W.Workload, gemm=A.AFD_GEMM_TENSOR, layers=None, stream=None,
                 max_total_tokens=0, wait_timeout_ns=0, device="cuda", flags=0, ring_depth=1,
                 canary=False):
        import torch
        self.w = w
        self.device = device
        self.layers = w.layers if layers is None else layers
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        self.cfg = A.make_config(w.num_peers, w.token_cap, w.hidden, w.num_experts, w.topk,
                                 w.inter, w.shared_inter, act=w.act, renorm=w.renorm,
                                 routed_scaling=w.routed_scaling, max_layers=self.layers,
                                 max_total_tokens=max_total_tokens, gemm=gemm,
                                 wait_timeout_ns=wait_timeout_ns,
                                 flags=flags | (A.AFD_CFG_CANARY if canary else 0),
                                 ring_depth=ring_depth)
        self.ctx = A.afd_create(self.cfg, self.stream.cuda_stream)
        self.layout = A.afd_slot_layout(self.cfg)
        self.canary = bool(canary)
        self.host = W.host_inputs(w)
        self.x = [act_tensor(a, w.act, device) for a in self.host["x"]]
        self.Wg = torch.from_numpy(self.host["Wg"]).to(device)
        self.bias = None if self.host["bias"] is None else torch.from_numpy(self.host["bias"]).to(device)
        self.weights = []
        for layer in range(self.layers):
            wt = W.expert_weights(w, layer, device)
            self.weights.append(wt)
            A.afd_set_layer(self.ctx, layer, self.Wg.data_ptr(),
                            self.bias.data_ptr() if self.bias is not None else 0,
                            wt["W13"].data_ptr(), wt["Wd"].data_ptr(),
                            wt["W13s"].data_ptr() if wt["W13s"] is not None else 0,
                            wt["Wds"].data_ptr() if wt["Wds"] is not None else 0)
        self.seq = 0
        self.last_seq = {}
        dt = torch.bfloat16 if w.act == "bf16" else torch.float32
        self.out = [torch.empty((max(n, 1), w.hidden), dtype=dt, device=device) for n in w.seq_lens]
        self.batched = True  # pack / unpack all listed peers in one call (afd_pack_slots / afd_unpack_splits)

    # -- attention side, simulated ------------------------------------------------
    def pack_all(self, layer=0, stage=0, peers=None, with_shared=None):
        ws = (self.w.shared_inter > 0) if with_shared is None else with_shared
        peers = list(range(self.w.num_peers)) if peers is None else list(peers)
        if self.batched:
            seqs = [self.seq + 1 + i for i in range(len(peers))]
            ns = [self.w.seq_lens[p] for p in peers]
            rc = A.afd_pack_slots(self.ctx, peers, stage, layer,
                                  [self.x[p].data_ptr() if n else 0 for p, n in zip(peers, ns)], ns, ws, seqs)
            if rc:
                raise A.AfdError(rc, "afd_pack_slots")
            self.seq += len(peers)
            for p, s in zip(peers, seqs):
                self.last_seq[(p, stage)] = s
            return
        for p in peers:
            self.seq += 1
            n = self.w.seq_lens[p]
            rc = A.afd_pack_slot(self.ctx, p, stage, layer, self.x[p].data_ptr() if n else 0, n,
                                 ws, self.seq)
            if rc:
                raise A.AfdError(rc, "afd_pack_slot")
            self.last_seq[(p, stage)] = self.seq

    def forward(self, layer=0, stage=0, slots=None):
        slots = list(range(self.w.num_peers)) if slots is None else list(slots)
        lens = [self.w.seq_lens[p] for p in slots]
        return A.afd_ffn_forward(self.ctx, layer, stage, lens, slots)

    def unpack_all(self, stage=0, peers=None):
        peers = list(range(self.w.num_peers)) if peers is None else list(peers)
        if self.batched:
            ns = [self.w.seq_lens[p] for p in peers]
            rc = A.afd_unpack_splits(self.ctx, peers, stage,
                                     [self.out[p].data_ptr() if n else 0 for p, n in zip(peers, ns)], ns,
                                     [self.last_seq[(p, stage)] for p in peers])
            if rc:
                raise A.AfdError(rc, "afd_unpack_splits")
            return self.out
        for p in peers:
            n = self.w.seq_lens[p]
            rc = A.afd_unpack_split(self.ctx, p, stage, self.out[p].data_ptr() if n else 0, n,
                                    self.last_seq[(p, stage)])
            if rc:
                raise A.AfdError(rc, "afd_unpack_split")
        return self.out

    # -- grouped form: the Attention side routes ---------------------------------
    def prepare_grouped(self, seed=0):
        """Draw the Attention side's routing (distinct top-k experts per token,
        seeded) and build each peer's routed rows grouped by expert (stable
        sort of the flattened ids) and its group list, on the device."""
        import torch
        w = self.w
        rng = np.random.default_rng(seed)
        self.g_rows, self.g_list, self.g_n = [], [], []
        for p, n in enumerate(w.seq_lens):
            ids = np.argsort(rng.random((n, w.num_experts)), axis=1)[:, :w.topk]
            order = np.argsort(ids.reshape(-1), kind="stable")
            rows = np.ascontiguousarray(self.host["x"][p][order // w.topk])
            self.g_rows.append(act_tensor(rows, w.act, self.device) if rows.shape[0] else None)
            self.g_list.append(np.bincount(ids.reshape(-1), minlength=w.num_experts))
            self.g_n.append(int(rows.shape[0]))
        dt = torch.bfloat16 if w.act == "bf16" else torch.float32
        self.g_y = [torch.empty((max(r, 1), w.hidden), dtype=dt, device=self.device) for r in self.g_n]

    def pack_grouped_all(self, layer=0, stage=0, with_shared=None):
        ws = (self.w.shared_inter > 0) if with_shared is None else with_shared
        for p, n in enumerate(self.w.seq_lens):
            self.seq += 1
            rows = self.g_rows[p]
            rc = A.afd_pack_grouped(self.ctx, p, stage, layer, rows.data_ptr() if rows is not None else 0,
                                    self.g_n[p], self.g_list[p], self.x[p].data_ptr() if n else 0, n,
                                    ws, self.seq)
            if rc:
                raise A.AfdError(rc, "afd_pack_grouped")
            self.last_seq[(p, stage)] = self.seq

    def forward_grouped(self, layer=0, stage=0):
        slots = list(range(self.w.num_peers))
        return A.afd_ffn_forward_grouped(self.ctx, layer, stage, self.g_n, list(self.w.seq_lens), slots)

    def unpack_grouped_all(self, stage=0, with_shared=None):
        ws = (self.w.shared_inter > 0) if with_shared is None else with_shared
        for p, n in enumerate(self.w.seq_lens):
            rc = A.afd_unpack_grouped(self.ctx, p, stage, self.g_y[p].data_ptr() if self.g_n[p] else 0,
                                      self.g_n[p], self.out[p].data_ptr() if (ws and n) else 0, n,
                                      self.last_seq[(p, stage)])
            if rc:
                raise A.AfdError(rc, "afd_unpack_grouped")
        return self.g_y, self.out

    def poll(self):
        return A.afd_poll_status(self.ctx)

    # -- inspection -----------------------------------------------------------------
    def window(self, direction):
        ptr, n = A.afd_get_window(self.ctx, direction)
        return device_view(ptr, n)

    def workspace(self, which, nbytes=None):
        ptr, cap = A.afd_get_workspace(self.ctx, which)
        return device_view(ptr, cap if nbytes is None else nbytes)

    def weights_numpy(self, layer):
        d = W.weights_to_numpy(self.weights[layer])
        d["Wg"] = self.host["Wg"]
        d["bias"] = self.host["bias"]
        return d

    def close(self):
        if self.ctx:
            A.afd_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class RankSet:
    """Token-level dispatch on one GPU: ffn_size FFN-rank contexts, each with
    its block of the experts (a view into the layer's expert weights, no
    copy) and the shared expert, and one Attention-peer object per peer that
    sends to all of them.  The Attention side's gate is the library's router
    (afd_route_noalloc) on each peer's tokens.  Torch plumbing only."""

    def __init__(self, w: W.Workload, ffn_size, ring_depth=1, gemm=A.AFD_GEMM_TENSOR, layers=None,
                 multiplier=2.0, wait_timeout_ns=0, max_total_tokens=0, device="cuda"):
        import torch
        self.w, self.F, self.device = w, ffn_size, device
        self.layers = w.layers if layers is None else layers
        self.stream = torch.cuda.current_stream()
        self.host = W.host_inputs(w)
        self.x = [act_tensor(a, w.act, device) for a in self.host["x"]]
        self.Wg = torch.from_numpy(self.host["Wg"]).to(device)
        self.bias = None if self.host["bias"] is None else torch.from_numpy(self.host["bias"]).to(device)
        self.weights = [W.expert_weights(w, layer, device) for layer in range(self.layers)]
        self.ranks, self.experts, self.cfgs = [], [], []
        for r in range(ffn_size):
            first, cnt = A.afd_expert_range(w.num_experts, ffn_size, r)
            cfg = A.make_config(w.num_peers, w.token_cap, w.hidden, cnt, w.topk, w.inter,
                                w.shared_inter, act=w.act, renorm=w.renorm,
                                routed_scaling=w.routed_scaling, ring_depth=ring_depth,
                                max_total_tokens=max_total_tokens or w.total_tokens,
                                max_layers=self.layers, gemm=gemm,
                                routed_cap_multiplier=multiplier,
                                wait_timeout_ns=wait_timeout_ns, ffn_rank=r, ffn_size=ffn_size)
            ctx = A.afd_create(cfg, self.stream.cuda_stream)
            for layer, wt in enumerate(self.weights):
                W13, Wd = wt["W13"], wt["Wd"]
                A.afd_set_layer(ctx, layer, 0, 0, W13[first].data_ptr(), Wd[first].data_ptr(),
                                wt["W13s"].data_ptr() if wt["W13s"] is not None else 0,
                                wt["Wds"].data_ptr() if wt["Wds"] is not None else 0)
            self.ranks.append(ctx)
            self.experts.append((first, cnt))
            self.cfgs.append(cfg)
        self.attn = [A.afd_attn_create(self.ranks, p, w.num_experts, self.stream.cuda_stream)
                     for p in range(w.num_peers)]
        dt = torch.bfloat16 if w.act == "bf16" else torch.float32
        self.out = [torch.empty((max(n, 1), w.hidden), dtype=dt, device=device) for n in w.seq_lens]
        self.ids = [torch.zeros((max(n, 1), w.topk), dtype=torch.int32, device=device)
                    for n in w.seq_lens]
        self.wts = [torch.zeros((max(n, 1), w.topk), dtype=torch.float32, device=device)
                    for n in w.seq_lens]
        self.seq = 0
        self.last_seq = {}

    def route(self):
        """The Attention side's gate on every peer's tokens."""
        w = self.w
        for p, n in enumerate(w.seq_lens):
            if not n:
                continue
            rc = A.afd_route_noalloc(self.x[p].data_ptr(), n, w.hidden,
                                     A.AFD_DTYPE_BF16 if w.act == "bf16" else A.AFD_DTYPE_F32,
                                     self.Wg.data_ptr(),
                                     self.bias.data_ptr() if self.bias is not None else 0,
                                     w.num_experts, w.topk, w.renorm, w.routed_scaling,
                                     self.ids[p].data_ptr(), self.wts[p].data_ptr(),
                                     self.stream.cuda_stream)
            if rc:
                raise A.AfdError(rc, "afd_route_noalloc")

    def dispatch_all(self, stage=0, layer=0, with_shared=None):
        ws = (self.w.shared_inter > 0) if with_shared is None else with_shared
        for p, n in enumerate(self.w.seq_lens):
            self.seq += 1
            rc = A.afd_attn_dispatch(self.attn[p], stage, layer, self.x[p].data_ptr() if n else 0,
                                     n, self.ids[p].data_ptr() if n else 0, ws, self.seq)
            if rc:
                raise A.AfdError(rc, "afd_attn_dispatch")
            self.last_seq[(p, stage)] = self.seq

    def serve_all(self, n_items=1, ranks=None):
        slots = list(range(self.w.num_peers))
        for r in (range(self.F) if ranks is None else ranks):
            rc = A.afd_ffn_serve(self.ranks[r], slots, n_items, A.AFD_FORM_GROUPED)
            if rc:
                raise A.AfdError(rc, "afd_ffn_serve")

    def combine_all(self, stage=0):
        for p, n in enumerate(self.w.seq_lens):
            rc = A.afd_attn_combine(self.attn[p], stage, self.wts[p].data_ptr() if n else 0,
                                    self.out[p].data_ptr() if n else 0, n,
                                    self.last_seq[(p, stage)])
            if rc:
                raise A.AfdError(rc, "afd_attn_combine")
        return self.out

    def poll(self):
        """(first status of the ranks, of the peers)"""
        fr = next((s for s in (A.afd_poll_status(c) for c in self.ranks) if s), 0)
        fa = next((s for s in (A.afd_attn_poll_status(a) for a in self.attn) if s), 0)
        return fr, fa

    def window(self, r, direction):
        ptr, n = A.afd_get_window(self.ranks[r], direction)
        return device_view(ptr, n)

    def rank_weights_numpy(self, r, layer=0):
        first, cnt = self.experts[r]
        d = W.weights_to_numpy(self.weights[layer])
        d["W13"] = np.ascontiguousarray(d["W13"][first:first + cnt])
        d["Wd"] = np.ascontiguousarray(d["Wd"][first:first + cnt])
        d["Wg"] = None
        d["bias"] = None
        return d

    def close(self):
        for a in self.attn:
            A.afd_attn_destroy(a)
        self.attn = []
        for c in self.ranks:
            A.afd_destroy(c)
        self.ranks = []
