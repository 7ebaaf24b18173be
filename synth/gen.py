"""Input generation for the scaled GEMM: seeded normals, quantised to e4m3.

The recipe (the pages give shapes and distributions, not values):
  * one ``torch.Generator('cpu')`` per case, seeded with the case's seed; A is
    drawn first, then B, as float32 ``randn`` times the case's standard
    deviation (N(0,1) for A, N(0,1) or N(0,0.02) for B);
  * ptpc:        A quantised per row (per token), B per output row (per
    channel), scale = amax / 448, codes = RNE(x / scale) clamped to +-448;
  * blockscale:  A per 1x128 block along K, B per 128x128 block, fp32 scales,
    same rule;
  * mxfp8:       per 32 consecutive K elements of a row, scale 2^e with
    e = ceil(log2(amax / 448)) stored as e8m0 code e + 127 (clamped to 0..254);
  * an all-zero row / block gets scale 1.0 (e8m0 127);
  * bf16:        randn rounded to bf16 (RNE).
Scale layouts: ptpc sa [M], sb [N]; blockscale sa [K/128, M] (K-block major),
sb [ceil(N/128), K/128]; mxfp8 sa [K/32, M], sb [K/32, N] (K-block major).
"""
import dataclasses
import math
from typing import Optional

import numpy as np
import torch

E4M3_MAX = 448.0


@dataclasses.dataclass
class Case:
    """One GEMM problem.  Tensors are CPU torch tensors.

    A, B:  uint8 e4m3 codes [M,K] / [N,K] (bf16 mode: torch.bfloat16)
    sa, sb: scales in the layout of the mode (None for bf16)
    """

    mode: str
    M: int
    N: int
    K: int
    A: torch.Tensor
    B: torch.Tensor
    sa: Optional[torch.Tensor]
    sb: Optional[torch.Tensor]
    seed: int = 0

    def numpy(self):
        """(A, B, sa, sb) as numpy arrays in the oracle's conventions."""
        if self.mode == "bf16":
            A = self.A.view(torch.int16).numpy().view(np.uint16)
            B = self.B.view(torch.int16).numpy().view(np.uint16)
            return A, B, None, None
        return self.A.numpy(), self.B.numpy(), self.sa.numpy(), self.sb.numpy()

    @property
    def flops(self) -> float:
        return gemm_flops(self.M, self.N, self.K)


def _to_e4m3_codes(x: torch.Tensor) -> torch.Tensor:
    return x.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)


def _safe_scale(amax: torch.Tensor) -> torch.Tensor:
    s = amax / E4M3_MAX
    return torch.where(amax > 0, s, torch.ones_like(s))


def quantize_e4m3_rows(x: torch.Tensor):
    """Per-row amax/448 quantisation: returns (codes uint8 [R,C], scale fp32 [R])."""
    x = x.float()
    s = _safe_scale(x.abs().amax(dim=1))
    return _to_e4m3_codes(x / s[:, None]), s.contiguous()


def quantize_e4m3_blocks_1x128(x: torch.Tensor):
    """A-side blockscale: one scale per row per 128 K.  Returns codes, scale [K/128, M]."""
    R, C = x.shape
    assert C % 128 == 0
    xb = x.float().reshape(R, C // 128, 128)
    s = _safe_scale(xb.abs().amax(dim=2))  # [R, K/128]
    q = _to_e4m3_codes(xb / s[:, :, None]).reshape(R, C)
    return q, s.t().contiguous()


def quantize_e4m3_blocks_128x128(w: torch.Tensor):
    """B-side blockscale: one scale per 128x128 block.  Returns codes, scale [ceil(N/128), K/128]."""
    N, K = w.shape
    assert K % 128 == 0
    nb = (N + 127) // 128
    wp = torch.zeros(nb * 128, K, dtype=torch.float32)
    wp[:N] = w.float()
    wb = wp.reshape(nb, 128, K // 128, 128)
    s = _safe_scale(wb.abs().amax(dim=(1, 3)))  # [nb, K/128]
    q = _to_e4m3_codes(wb / s[:, None, :, None]).reshape(nb * 128, K)[:N]
    return q.contiguous(), s.contiguous()


def quantize_mx_rows(x: torch.Tensor):
    """MX quantisation per 32 K elements of each row.  Returns codes, e8m0 codes [K/32, R]."""
    R, C = x.shape
    assert C % 32 == 0
    xb = x.float().reshape(R, C // 32, 32)
    amax = xb.abs().amax(dim=2).double()
    e = torch.ceil(torch.log2(amax / E4M3_MAX))
    e = torch.where(amax > 0, e, torch.zeros_like(e))
    code = (e + 127).clamp(0, 254)
    scale = torch.pow(2.0, code - 127).float()
    q = _to_e4m3_codes(xb / scale[:, :, None]).reshape(R, C)
    return q, code.to(torch.uint8).t().contiguous()


def _draw(gen, rows, cols, std):
    return torch.randn(rows, cols, generator=gen, dtype=torch.float32) * std


_QUANT_A = {
    "ptpc": quantize_e4m3_rows,
    "blockscale": quantize_e4m3_blocks_1x128,
    "mxfp8": quantize_mx_rows,
}
_QUANT_B = {
    "ptpc": quantize_e4m3_rows,
    "blockscale": quantize_e4m3_blocks_128x128,
    "mxfp8": quantize_mx_rows,
}


def make_case(mode: str, M: int, N: int, K: int, seed: int = 0, a_std: float = 1.0, b_std: float = 1.0,
              cache: Optional[dict] = None) -> Case:
    """Seeded synthetic case in the given scale mode (A drawn first, then B).

    ``cache`` (optional dict) reuses the quantised A and the generator state
    after A between cases that share (mode, M, K, seed, a_std): the values are
    exactly those of a fresh draw.
    """
    if mode not in ("bf16",) and mode not in _QUANT_A:
        raise ValueError("unknown mode %r" % mode)
    key = (mode, M, K, seed, a_std)
    if cache is not None and key in cache:
        qa, sa, state = cache[key]
        g = torch.Generator("cpu")
        g.set_state(state)
    else:
        g = torch.Generator("cpu")
        g.manual_seed(seed)
        a = _draw(g, M, K, a_std)
        if mode == "bf16":
            qa, sa = a.bfloat16().contiguous(), None
        else:
            qa, sa = _QUANT_A[mode](a)
            qa = qa.contiguous()
        del a
        if cache is not None:
            cache[key] = (qa, sa, g.get_state())
    b = _draw(g, N, K, b_std)
    if mode == "bf16":
        return Case(mode, M, N, K, qa, b.bfloat16().contiguous(), None, None, seed)
    qb, sb = _QUANT_B[mode](b)
    return Case(mode, M, N, K, qa, qb.contiguous(), sa, sb, seed)


def make_int_case(M: int, N: int, K: int, lo: int = -16, hi: int = 16, seed: int = 0) -> Case:
    """ptpc case with integer-valued e4m3 operands in [lo, hi] and unit scales."""
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    a = torch.randint(lo, hi + 1, (M, K), generator=g).float()
    b = torch.randint(lo, hi + 1, (N, K), generator=g).float()
    return Case(
        "ptpc", M, N, K, _to_e4m3_codes(a), _to_e4m3_codes(b),
        torch.ones(M, dtype=torch.float32), torch.ones(N, dtype=torch.float32), seed,
    )


def with_extreme_mx_codes(case: Case, seed: int = 0, codes=(0, 1, 127, 253, 254)) -> Case:
    """The same mxfp8 operands with e8m0 scale codes at the ends of the range,
    mixed per K block: block j of A takes a base code a_j drawn from `codes`, each
    row of the block a_j + d (d in {-1, 0, 1}, kept in [0, 254]); block j of B
    takes 254 - a_j + e (e in {-1, 0, 1}, kept in [0, 254]).  Every block's
    product of scales is then 2^-2 .. 2^2, so all blocks contribute to every
    output element while the tensor core decodes codes 0, 1, 253 and 254."""
    assert case.mode == "mxfp8"
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    kb = case.K // 32
    base = torch.tensor(codes, dtype=torch.int64)[torch.randint(0, len(codes), (kb,), generator=g)]
    da = torch.randint(-1, 2, (kb, case.M), generator=g)
    db = torch.randint(-1, 2, (kb, case.N), generator=g)
    sa = (base[:, None] + da).clamp(0, 254).to(torch.uint8).contiguous()
    sb = (254 - base[:, None] + db).clamp(0, 254).to(torch.uint8).contiguous()
    return dataclasses.replace(case, sa=sa, sb=sb)


def with_wide_block_scales(case: Case, seed: int = 0, lo: int = -40, hi: int = 40, zero_frac: float = 0.05) -> Case:
    """The same blockscale operands with fp32 block scales spread over binades
    2^lo .. 2^hi (a random significand in [1, 2) times 2^u, u uniform in [lo, hi],
    random sign), a fraction `zero_frac` of them set to zero, plus one A row and
    one B block column of scales that are all zero."""
    assert case.mode == "blockscale"
    g = torch.Generator("cpu")
    g.manual_seed(seed)

    def draw(shape):
        sig = 1.0 + torch.rand(shape, generator=g, dtype=torch.float64)
        u = torch.randint(lo, hi + 1, shape, generator=g).double()
        sign = torch.where(torch.rand(shape, generator=g) < 0.5, -1.0, 1.0).double()
        v = (sign * sig * torch.pow(2.0, u)).float()
        return torch.where(torch.rand(shape, generator=g) < zero_frac, torch.zeros_like(v), v)

    sa = draw(tuple(case.sa.shape))
    sb = draw(tuple(case.sb.shape))
    sa[:, case.M // 2] = 0.0          # one row of A: every block scale zero
    sb[:, sb.shape[1] // 2] = 0.0     # one K block of B: zero for every N block
    return dataclasses.replace(case, sa=sa.contiguous(), sb=sb.contiguous())


@dataclasses.dataclass
class GatherCase:
    """One gather-GEMM problem (ptpc): output row i reads row idx[i] of A_src.

    A_src uint8 e4m3 [R, K] with per-row scales sa_src fp32 [R]; idx int32 [M];
    B uint8 e4m3 [N, K] with per-channel scales sb fp32 [N]."""

    M: int
    N: int
    K: int
    R: int
    A_src: torch.Tensor
    sa_src: torch.Tensor
    idx: torch.Tensor
    B: torch.Tensor
    sb: torch.Tensor
    seed: int = 0
    mode: str = "ptpc"

    def numpy(self):
        """(A_src, idx, B, sa_src, sb) as numpy arrays."""
        return self.A_src.numpy(), self.idx.numpy(), self.B.numpy(), self.sa_src.numpy(), self.sb.numpy()

    @property
    def flops(self) -> float:
        return gemm_flops(self.M, self.N, self.K)


def paged_indices(M: int, R: int, page: int, g: torch.Generator, min_len: int = 64, max_len: int = 2048) -> torch.Tensor:
    """Row indices of M tokens read from a paged cache of R rows: sequences of
    lengths drawn uniformly from [min_len, max_len] (the last one cut to fit),
    each stored in pages of `page` rows taken from a shuffled free list, read in
    order.  int32 [M]."""
    free = torch.randperm(R // page, generator=g)
    out, used, left = [], 0, M
    while left > 0:
        n = min(left, int(torch.randint(min_len, max_len + 1, (1,), generator=g)))
        npages = (n + page - 1) // page
        if used + npages > free.numel():
            raise ValueError("cache of %d rows too small for %d gathered rows" % (R, M))
        pages = free[used:used + npages]
        used += npages
        out.append((pages[:, None] * page + torch.arange(page)[None, :]).reshape(-1)[:n])
        left -= n
    return torch.cat(out).to(torch.int32).contiguous()


def make_gather_case(M: int, R: int, N: int, K: int, seed: int = 0, b_std: float = 0.02,
                     page: int = 64) -> GatherCase:
    """Seeded gather-GEMM case: A_src ~ N(0,1) [R, K] quantised per row, B ~ N(0, b_std)
    [N, K] quantised per output channel (drawn in that order), then paged indices."""
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    qa, sa = quantize_e4m3_rows(_draw(g, R, K, 1.0))
    qb, sb = quantize_e4m3_rows(_draw(g, N, K, b_std))
    idx = paged_indices(M, R, page, g)
    return GatherCase(M, N, K, R, qa.contiguous(), sa, idx, qb.contiguous(), sb, seed)


# The gather-GEMM workload: a KV projection of 32 heads x (128 + 128) columns over
# a 512-wide latent, for 16384 tokens gathered from a 65536-row paged cache.
GATHER_CONFIGS = {
    "g_ptpc_gather_16384x8192x512": (16384, 65536, 8192, 512, 0),
}


def gemm_flops(M, N, K) -> float:
    return 2.0 * M * N * K


def gemm_bytes(mode, M, N, K) -> float:
    """Algorithmic bytes of one GEMM: operands once, C once, scales once."""
    el = 2 if mode == "bf16" else 1
    b = el * (M * K + N * K) + 2 * M * N
    if mode == "ptpc":
        b += 4 * (M + N)
    elif mode == "blockscale":
        b += 4 * (M * (K // 128) + math.ceil(N / 128) * (K // 128))
    elif mode == "mxfp8":
        b += (M + N) * (K // 32)
    return float(b)


# The five workloads, as (name, mode, M, N, K, seed, a_std, b_std).
CONFIGS = {
    "c0_ptpc_256x512x256": ("ptpc", 256, 512, 256, 0, 1.0, 1.0),
    "c1_ptpc_4096x7168x256": ("ptpc", 4096, 7168, 256, 0, 1.0, 1.0),
    "c2_ptpc_16384x7168x512": ("ptpc", 16384, 7168, 512, 0, 1.0, 0.02),
    "c2_ptpc_32768x7168x1792": ("ptpc", 32768, 7168, 1792, 0, 1.0, 0.02),
    "c3_blockscale_16384x7168x2048": ("blockscale", 16384, 7168, 2048, 0, 1.0, 0.02),
    "c3_mxfp8_32768x7168x1792": ("mxfp8", 32768, 7168, 1792, 0, 1.0, 0.02),
    "c4_ptpc_32768x6288x7168": ("ptpc", 32768, 6288, 7168, 0, 1.0, 0.02),
    "c4_ptpc_32768x3648x7168": ("ptpc", 32768, 3648, 7168, 0, 1.0, 0.02),
    "c4_ptpc_32768x6400x7168": ("ptpc", 32768, 6400, 7168, 0, 1.0, 0.02),
    "c4_bf16_4096x896x1024": ("bf16", 4096, 896, 1024, 233, 1.0, 1.0),
    # mxfp8 on the blockscale workload's shape (the second shape the pages run the
    # block-scaled modes at); a parity case and a separate bench line, not a suite step
    "x_mxfp8_16384x7168x2048": ("mxfp8", 16384, 7168, 2048, 0, 1.0, 0.02),
}

# One benchmark step runs each of these once (every M x 7168 x K shape, all
# three scale modes, the unpadded-N shapes and the BF16 GEMM).
SUITE = [k for k in CONFIGS if k[:3] in ("c1_", "c2_", "c3_", "c4_")]
# Further shapes: checked at full size and timed on their own.
EXTRA = [k for k in CONFIGS if k.startswith("x_")]
