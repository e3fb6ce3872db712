"""A seeded workload resident on the GPU: x, router weight and bias from the
shared generator, expert master weights generated in place on the device and
encoded by the library's own block quantiser (moe_quantize), scales in the
TILED layout the expert GEMMs read.  Used by the GPU tests, the smoke check
and the benchmark; the oracle side regenerates the same inputs on the host.
"""
from __future__ import annotations

import numpy as np

import synth


def workload(spec) -> dict:
    return synth.workload_spec(spec)


class GpuWorkload:
    def __init__(self, spec, torch, device="cuda", cap=10.0, mx_scale_mode=0, chunk_experts=8,
                 with_weights=True, act_static=None, bias_in_weights=0, routed_scale=1.0, ffn_schedule=0,
                 y_format=None):
        import block_scaled_fp4_route_gb300 as moe
        self.torch = torch
        self.moe = moe
        self.w = w = workload(spec)
        T, H, E, k, F = w["T"], w["H"], w["E"], w["k"], w["F"]
        self.fmt = w["fmt"]
        # act_static: NVFP4 static activation globals fp32 [E, 2] (numpy), or None
        self.act_static = None if act_static is None else torch.from_numpy(
            np.ascontiguousarray(act_static, np.float32)).to(device)
        self.route_opts = dict(bias_in_weights=bool(bias_in_weights), routed_scale=float(routed_scale))
        self.cfg = moe.make_config(T, H, E, k, F, w["fmt"], swiglu_cap=cap, mx_scale_mode=mx_scale_mode,
                                   act_global_mode=0 if act_static is None else 1,
                                   bias_in_weights=int(bias_in_weights), routed_scale=routed_scale,
                                   ffn_schedule=ffn_schedule, y_format=y_format)
        self.x = synth.dev_x(w, torch, device)
        self.w_router = synth.dev_router_weight(w, torch, device)
        self.bias = torch.from_numpy(synth.router_bias(w)).to(device)
        self.ws = torch.empty(moe.moe_workspace_size(self.cfg), dtype=torch.uint8, device=device)
        self.layout = moe.moe_workspace_layout(self.cfg)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        self.mats = {}
        if with_weights:
            for which, N, K in (("gate", F, H), ("up", F, H), ("down", H, F)):
                self.mats[which] = self._encode(which, N, K, chunk_experts, mx_scale_mode, device)
        self.qw = {k_: moe.qweight(*v) for k_, v in self.mats.items()}

    def _encode(self, which, N, K, chunk, mx_mode, device):
        torch, moe, w = self.torch, self.moe, self.w
        E = w["E"]
        nv = self.fmt == "nvfp4"
        cb = K // 2 if nv else K
        bs = 16 if nv else 32
        codes = torch.empty((E, N, cb), dtype=torch.uint8, device=device)
        scales = torch.empty((E, N, K // bs), dtype=torch.uint8, device=device)
        glob = torch.empty(E, dtype=torch.float32, device=device) if nv else None
        buf = torch.empty((min(chunk, E), N, K), dtype=torch.float32, device=device)
        for e0 in range(0, E, chunk):
            ne = min(chunk, E - e0)
            m = synth.dev_expert_matrices(w, which, e0, ne, torch, out=buf[:ne])
            moe.moe_quantize(self.fmt, m.view(ne * N, K), codes[e0:e0 + ne], scales[e0:e0 + ne],
                             glob[e0:e0 + ne] if nv else None, group_rows=N if nv else 0,
                             layout=moe.SCALES_TILED, mx_scale_mode=mx_mode)
        del buf
        return codes, scales, glob

    def weight_bytes(self, touched_experts=None) -> int:
        """Bytes of the encoded expert weights (codes + scales + globals)."""
        tot = 0
        for codes, scales, glob in self.mats.values():
            per = (codes[0].numel() + scales[0].numel() + (4 if glob is not None else 0))
            tot += per * (self.w["E"] if touched_experts is None else touched_experts)
        return tot

    def forward(self, stream=None):
        self.moe.moe_forward(self.cfg, self.x, self.w_router, self.bias, self.qw["gate"], self.qw["up"],
                             self.qw["down"], self.out, self.ws, stream, act_static_scales=self.act_static)
        return self.out

    def ws_view(self, name, dtype, count):
        """A typed view of one intermediate buffer of the workspace."""
        torch = self.torch
        off = self.layout[name]
        item = torch.empty((), dtype=dtype).element_size()
        return self.ws[off:off + count * item].view(dtype)

    def y_raw(self):
        """The workspace's expert output rows as bytes (moe_y_bytes of the config)."""
        off = self.layout["y_perm"]
        return self.ws[off:off + self.moe.moe_y_bytes(self.cfg)]

    def routing(self):
        """topk idx / w, counts, offsets, perm, pair_pos, seg_start from the workspace (numpy)."""
        torch = self.torch
        T, k, E = self.w["T"], self.w["k"], self.w["E"]
        P = T * k
        g = lambda n, dt, c: self.ws_view(n, dt, c).cpu().numpy()
        return dict(idx=g("topk_idx", torch.int32, P).reshape(T, k), w=g("topk_w", torch.float32, P).reshape(T, k),
                    counts=g("counts", torch.int32, E), offsets=g("offsets", torch.int32, E + 1),
                    perm=g("perm", torch.int32, P), pair_pos=g("pair_pos", torch.int32, P).reshape(T, k),
                    seg_start=g("seg_start", torch.int32, E + 1))


def untile_scales(tiled: np.ndarray, rows: int, cols: int, tile_rows: int = 128) -> np.ndarray:
    """Scale atoms (moe.h) -> row-major [rows, cols].  tile_rows = 128 is the
    TILED weight layout; 64 is the activation layout of the workspace."""
    r = np.arange(rows)[:, None]
    c = np.arange(cols)[None, :]
    rr = r % tile_rows
    off = ((r // tile_rows) * (cols >> 2) + (c >> 2)) * 512 + (rr & 31) * 16 + ((rr >> 5) & 3) * 4 + (c & 3)
    return np.asarray(tiled).reshape(-1)[off]
