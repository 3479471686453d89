"""Seeded synthetic inputs for the decode step (no decode-step arithmetic here).

This module only draws random inputs: sequence lengths, shuffled block tables,
KV pools, queries, new K/V rows, logits and per-request sampler settings.  It is
shared by the CUDA path's tests/benchmark and by the oracle checks; it computes
nothing the decode step computes (no append, no gather, no softmax, no filter).

The five workloads follow the shapes the pages discuss: the lab's tiny engine
(2 heads of dim 4, blocks of 4 tokens, a pool of 12 blocks, a 22-token
vocabulary; "Bai Lab tong hop -- Inference Engineering", configuration section),
Llama-style GQA with 8 KV heads and 16-token blocks ("Suy luan & Toi uu hoa
(Inference)" sections 3.1-3.2), long contexts for split-KV, a large fragmented
batch, and a sampler stress batch over a 152064-token vocabulary.

Recipe (all seeds fixed; seed = 1000 + workload number):
* lengths: uniform integers in [len_lo, len_hi] (CPU torch generator);
* physical blocks: one global random permutation of the pool; sequence b takes
  the next ceil(L_b / BS) entries.  With pool_factor > 1 the pool holds
  ceil(pool_factor * needed) blocks and the unused ones are scattered holes;
* unused block-table entries are -1;
* q, K, V, k_new, v_new ~ N(0, 1), rounded to bf16 (round-to-nearest-even) when
  the workload is bf16; the whole pool is random, including slots past each
  sequence's length;
* logits ~ N(0, logit_std^2) float32 (workload 5: rows 0..B/2-1 get +12 on one
  random id over N(0, 1); the rest are N(0, 0.1^2));
* values are drawn by a torch generator on the target device (CPU or CUDA), so
  CPU- and CUDA-generated values differ; both sides of every comparison always
  receive the same tensors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

__all__ = ["DecodeWorkload", "WORKLOADS", "workload", "make_decode_inputs", "make_sampler_inputs",
           "kv_bytes", "step_bytes"]


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    number: int
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    block_size: int
    len_lo: int
    len_hi: int
    dtype: str                 # "f32" or "bf16" (q, K, V, output)
    vocab: int
    logit_std: float
    temperature: float
    top_k: int
    top_p: float
    pool_factor: float = 1.0   # physical pool size / blocks needed
    num_blocks: int = 0        # fixed pool size (0: derived from pool_factor)
    fixed_lens: tuple = ()     # explicit lengths (overrides len_lo/len_hi)
    sampler_stress: bool = False

    @property
    def seed(self) -> int:
        return 1000 + self.number

    @property
    def max_len(self) -> int:
        return max(self.fixed_lens) if self.fixed_lens else self.len_hi

    @property
    def max_blocks(self) -> int:
        return -(-self.max_len // self.block_size)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


WORKLOADS = {
    1: DecodeWorkload("tiny-lab-f32", 1, batch=2, n_q_heads=2, n_kv_heads=2, head_dim=4,
                      block_size=4, len_lo=9, len_hi=13, dtype="f32", vocab=22, logit_std=1.0,
                      temperature=0.8, top_k=5, top_p=0.9, num_blocks=12, fixed_lens=(9, 13)),
    2: DecodeWorkload("gqa-b64-32q8kv-d128-bs16-L512..4096", 2, batch=64, n_q_heads=32,
                      n_kv_heads=8, head_dim=128, block_size=16, len_lo=512, len_hi=4096,
                      dtype="bf16", vocab=128256, logit_std=2.0, temperature=0.7, top_k=50,
                      top_p=0.9),
    3: DecodeWorkload("longctx-b8-64q8kv-d128-bs16-L32K..128K", 3, batch=8, n_q_heads=64,
                      n_kv_heads=8, head_dim=128, block_size=16, len_lo=32768, len_hi=131072,
                      dtype="bf16", vocab=128256, logit_std=1.0, temperature=1e-3, top_k=0,
                      top_p=1.0),
    4: DecodeWorkload("frag-b512-32q8kv-d128-bs16-L128..1024", 4, batch=512, n_q_heads=32,
                      n_kv_heads=8, head_dim=128, block_size=16, len_lo=128, len_hi=1024,
                      dtype="bf16", vocab=32000, logit_std=1.5, temperature=1.0, top_k=0,
                      top_p=0.95, pool_factor=1.25),
    5: DecodeWorkload("sampler-b256-v152064", 5, batch=256, n_q_heads=0, n_kv_heads=0,
                      head_dim=0, block_size=0, len_lo=0, len_hi=0, dtype="f32", vocab=152064,
                      logit_std=1.0, temperature=1.0, top_k=0, top_p=1.0, sampler_stress=True),
}


def workload(number: int, **overrides) -> DecodeWorkload:
    """A named workload, optionally shrunk (e.g. batch=4, len_hi=300) for fast tests."""
    w = WORKLOADS[number]
    w = replace(w, **overrides) if overrides else w
    if not w.fixed_lens and w.len_hi and w.len_lo > w.len_hi:
        raise ValueError(f"len_lo {w.len_lo} > len_hi {w.len_hi}: override both")
    return w


def _cpu_gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _dev_gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _lengths(w: DecodeWorkload, g: torch.Generator) -> torch.Tensor:
    if w.fixed_lens:
        return torch.tensor(w.fixed_lens, dtype=torch.int32)
    return torch.randint(w.len_lo, w.len_hi + 1, (w.batch,), generator=g, dtype=torch.int64).to(torch.int32)


def _tables(w: DecodeWorkload, lens: torch.Tensor, g: torch.Generator):
    """Shuffled physical block assignment; returns (block_tables [B, max_blocks], num_blocks)."""
    bs = w.block_size
    need = [(-(-int(L) // bs)) for L in lens.tolist()]
    total = sum(need)
    if w.num_blocks:
        nb = w.num_blocks
    else:
        nb = max(1, math.ceil(w.pool_factor * total))
    assert nb >= total, "pool too small for the drawn lengths"
    perm = torch.randperm(nb, generator=g).to(torch.int32)
    tables = torch.full((w.batch, w.max_blocks), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(need):
        tables[b, :n] = perm[off:off + n]
        off += n
    return tables, nb


def _normal(shape, g, device, dtype):
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return x.to(dtype)


def make_decode_inputs(w: DecodeWorkload, device="cpu", with_logits: bool = True) -> dict:
    """All inputs of one decode step for workload w, placed on `device`.

    Keys: seq_lens [B] int32 (length AFTER the append), block_tables [B, max_blocks]
    int32, k_cache / v_cache [NB, Hkv, BS, D], q [B, Hq, D], k_new / v_new [B, Hkv, D],
    logits [B, V] f32, temperature [B] f32, top_k [B] int32, top_p [B] f32,
    seeds [B] int64 (uint64 bit patterns), offsets [B] int64, num_blocks (int).
    """
    g = _cpu_gen(w.seed)
    lens = _lengths(w, g)
    tables, nb = _tables(w, lens, g)
    dev = torch.device(device)
    gv = _dev_gen(w.seed + 1, dev)
    dt = w.torch_dtype
    B, Hq, Hkv, D, BS = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.block_size
    out = dict(
        seq_lens=lens.to(dev),
        block_tables=tables.to(dev),
        num_blocks=nb,
        k_cache=_normal((nb, Hkv, BS, D), gv, dev, dt),
        v_cache=_normal((nb, Hkv, BS, D), gv, dev, dt),
        q=_normal((B, Hq, D), gv, dev, dt),
        k_new=_normal((B, Hkv, D), gv, dev, dt),
        v_new=_normal((B, Hkv, D), gv, dev, dt),
    )
    if with_logits:
        out.update(_sampler_params_uniform(w, dev))
        out["logits"] = (torch.randn((B, w.vocab), generator=gv, device=dev, dtype=torch.float32)
                         * w.logit_std)
    return out


def _sampler_params_uniform(w: DecodeWorkload, dev) -> dict:
    B = w.batch
    return dict(
        temperature=torch.full((B,), w.temperature, dtype=torch.float32, device=dev),
        top_k=torch.full((B,), w.top_k, dtype=torch.int32, device=dev),
        top_p=torch.full((B,), w.top_p, dtype=torch.float32, device=dev),
        seeds=torch.arange(B, dtype=torch.int64, device=dev),
        offsets=torch.zeros(B, dtype=torch.int64, device=dev),
    )


def make_sampler_inputs(w: DecodeWorkload, device="cpu", batch: int | None = None,
                        vocab: int | None = None) -> dict:
    """Sampler-only inputs.  For the stress workload: half peaked rows (N(0,1) plus
    +12 on one random id), half flat rows (N(0, 0.1^2)); per-row T ~ U[0.5, 1.5],
    top_k from {0, 20, 50, 1000}, top_p from {0.8, 0.95, 1.0}, random 64-bit seeds.
    Other workloads: logits ~ N(0, logit_std^2) with the workload's fixed settings."""
    B = batch or w.batch
    V = vocab or w.vocab
    dev = torch.device(device)
    g = _cpu_gen(w.seed + 7)
    gv = _dev_gen(w.seed + 9, dev)
    if not w.sampler_stress:
        p = _sampler_params_uniform(replace(w, batch=B), dev)
        p["logits"] = torch.randn((B, V), generator=gv, device=dev, dtype=torch.float32) * w.logit_std
        return p
    half = B // 2
    logits = torch.randn((B, V), generator=gv, device=dev, dtype=torch.float32)
    logits[half:] *= 0.1
    spike = torch.randint(0, V, (half,), generator=g)
    logits[torch.arange(half, device=dev), spike.to(dev)] += 12.0
    temperature = 0.5 + torch.rand((B,), generator=g, dtype=torch.float32)
    ks = torch.tensor([0, 20, 50, 1000], dtype=torch.int32)
    ps = torch.tensor([0.8, 0.95, 1.0], dtype=torch.float32)
    top_k = ks[torch.randint(0, 4, (B,), generator=g)]
    top_p = ps[torch.randint(0, 3, (B,), generator=g)]
    seeds = torch.randint(-2**63, 2**63 - 1, (B,), generator=g, dtype=torch.int64)
    return dict(logits=logits, temperature=temperature.to(dev), top_k=top_k.to(dev),
                top_p=top_p.to(dev), seeds=seeds.to(dev),
                offsets=torch.zeros(B, dtype=torch.int64, device=dev))


def kv_bytes(w: DecodeWorkload, seq_lens) -> int:
    """KV bytes one attention pass must read: sum_b L_b * Hkv * D * 2 (K and V) * elem."""
    total = int(torch.as_tensor(seq_lens).to(torch.int64).sum())
    return total * w.n_kv_heads * w.head_dim * 2 * w.elem_bytes


def step_bytes(w: DecodeWorkload, seq_lens) -> dict:
    """Algorithmic HBM bytes of one decode step, per kernel family.

    attention: KV read + q read + out write + block-table entries read;
    append: k_new/v_new read + the same bytes written into the pools;
    sampler: logits read + 4 per-row parameters + seeds/offsets + token write."""
    sl = torch.as_tensor(seq_lens).to(torch.int64)
    e = w.elem_bytes
    B, Hq, Hkv, D, BS = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.block_size
    blocks = int(((sl + BS - 1) // BS).sum()) if BS else 0
    attn = kv_bytes(w, sl) + 2 * B * Hq * D * e + 4 * blocks + 4 * B
    append = 2 * (2 * B * Hkv * D * e) + 4 * B + 4 * B
    sampler = 4 * B * w.vocab + B * (4 + 4 + 4 + 8 + 8) + 4 * B
    return dict(attention=attn, append=append, sampler=sampler, total=attn + append + sampler)
