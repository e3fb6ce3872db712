"""MXFP8 KV-cache quantiser (moe_kv_quantize_mxfp8) against the oracle's MXFP8
quantiser along head_dim: codes and E8M0 scales bit-exact, on head_dim 64,
128 and 256, ragged token counts, a slot mapping into a larger cache (with
skipped padding tokens and untouched slots), a fused-projection token stride,
both scale modes, and blocks that are all zero, tiny or saturating."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import block_scaled_fp4_route_gb300 as moe  # noqa: E402


def kv_values(tokens, heads, head_dim, seed):
    """bf16 bits of seeded N(0,1) stand-ins with special blocks: all zero,
    tiny (2^-130: the E8M0 clamp), huge (x1e4) and the OCP floor rule's
    saturating case (a block maximum in (448, 512) times its scale)."""
    z = synth.normals(seed, synth.T_X, 0, tokens * heads * head_dim).reshape(tokens, heads, head_dim)
    z = z.astype(np.float32)
    nb = head_dim // 32
    flat = z.reshape(-1, 32)
    rng = np.random.default_rng(seed)
    pick = rng.choice(flat.shape[0], size=min(flat.shape[0], 4 * 4), replace=False)
    for i, b in enumerate(pick):
        kind = i % 4
        if kind == 0:
            flat[b] = 0.0
        elif kind == 1:
            flat[b] *= np.float32(2.0 ** -130)
        elif kind == 2:
            flat[b] *= np.float32(1e4)
        else:
            flat[b] = np.clip(flat[b], -1, 1)
            flat[b, 0] = np.float32(3.9)         # amax 3.9: scale 2^-7, 3.9 * 2^7 = 499 > 448 saturates
    bits = (flat.reshape(tokens, heads, head_dim).view(np.uint32) + 0x7FFF + ((flat.reshape(
        tokens, heads, head_dim).view(np.uint32) >> 16) & 1)) >> 16
    assert nb >= 1
    return bits.astype(np.uint16)


CASES = [  # tokens, heads, head_dim, slots ("none" | "perm" | "pad"), token stride factor, mode
    (1, 8, 128, "none", 1, 0),
    (37, 5, 64, "perm", 1, 0),
    (517, 8, 128, "pad", 1, 0),
    (300, 4, 256, "perm", 3, 0),        # K of a fused [tokens, 3, heads, head_dim] projection
    (129, 2, 256, "none", 1, 1),        # round-up scales (never saturate)
    (4096, 8, 128, "perm", 1, 0),
]


@pytest.mark.parametrize("tokens,heads,head_dim,slots,sf,mode", CASES)
def test_kv_quantize_bit_exact(tokens, heads, head_dim, slots, sf, mode):
    seed = 100 + tokens
    bits = kv_values(tokens, heads, head_dim, seed)
    stride = sf * heads * head_dim
    src = torch.zeros((tokens, stride), dtype=torch.int16)
    src[:, :heads * head_dim] = torch.from_numpy(bits.reshape(tokens, -1).view(np.int16))
    src = src.cuda().view(torch.bfloat16)
    kv = src[:, :heads * head_dim].view(tokens, heads, head_dim) if sf == 1 else \
        torch.as_strided(src, (tokens, heads, head_dim), (stride, head_dim, 1))
    rng = np.random.default_rng(seed)
    num_slots = tokens if slots == "none" else 2 * tokens + 3
    slot = None
    if slots != "none":
        slot = rng.permutation(num_slots)[:tokens].astype(np.int64)
        if slots == "pad":
            slot[rng.choice(tokens, size=tokens // 7, replace=False)] = -1
            slot[0] = num_slots + 5         # out of range: skipped as well
    codes = torch.full((num_slots, heads, head_dim), 0xAB, dtype=torch.uint8, device="cuda")
    scales = torch.full((num_slots, heads, head_dim // 32), 0xCD, dtype=torch.uint8, device="cuda")
    slot_t = None if slot is None else torch.from_numpy(slot).cuda()
    moe.moe_kv_quantize_mxfp8(kv, codes, scales, slots=slot_t, token_stride=stride, mx_scale_mode=mode)
    torch.cuda.synchronize()
    want_c, want_s = oracle.mxfp8_quantize(oracle.bf16_bits_to_f32(bits.reshape(-1, head_dim)), mode)
    want_c = want_c.reshape(tokens, heads, head_dim)
    want_s = want_s.reshape(tokens, heads, head_dim // 32)
    gc, gs = codes.cpu().numpy(), scales.cpu().numpy()
    dst = np.arange(tokens) if slot is None else slot
    live = (dst >= 0) & (dst < num_slots)
    assert np.array_equal(gc[dst[live]], want_c[live])
    assert np.array_equal(gs[dst[live]], want_s[live])
    untouched = np.ones(num_slots, bool)
    untouched[dst[live]] = False
    assert (gc[untouched] == 0xAB).all() and (gs[untouched] == 0xCD).all()
    # the special blocks were exercised
    assert (want_s == 0).any() and ((want_c.reshape(-1) & 0x7F) == 0x7E).any()


def test_kv_quantize_no_tokens_enqueues_nothing():
    codes = torch.zeros((4, 2, 64), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((4, 2, 2), dtype=torch.uint8, device="cuda")
    kv = torch.empty((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    moe.moe_kv_quantize_mxfp8(kv, codes, scales)
    torch.cuda.synchronize()
    assert int(codes.sum()) == 0
