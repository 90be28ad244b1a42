"""Seeded synthetic inputs for the FastOCR decode-attention path.

This module is shared by the CPU oracle's tests and by the CUDA path's tests and
benchmark. It holds NO arithmetic of the method: no softmax, no scoring, no
selection, no keep count. It only draws random K/V/q tensors, lays the KV cache
out in pages, and describes the workloads (shapes, keep ratio, schedule
lengths) so that both sides see byte-identical inputs.

Workloads (the shapes of the FastOCR pages' experiments, which run
Qwen2.5-VL-style decoders on dense document images, and of the Unlimited OCR
page's R-SWA decoder):

* ``tiny_f32``      -- 1 sequence, 2 layers, 4/2 heads, d=64, fp32, 16 prompt
                       tokens + a 16x16 image grid, 32 decode steps, tau=0.25.
* ``qwen7b_b1``     -- Qwen2.5-VL-7B attention shape (28 layers, 28 q heads,
                       4 KV heads, d=128), bf16, 64 prompt + 64x64 image,
                       512 decode steps, warm-up w=8, |C|=3, tau=0.05.
* ``serving_b32``   -- same attention shape, 32 sequences, 128 prompt +
                       128x64 image, 256 steps, random fixation start cells.
* ``multipage_b8``  -- 8 sequences, 4 image pages of 64x64 (16384 image
                       tokens), 64 prompt tokens, 4096 steps.
* ``rswa_b16``      -- DeepSeek-OCR-decoder-shaped MHA (12 layers, 10 heads,
                       d=128), bf16, 16 sequences, global prefix of
                       2560 visual + 64 prompt tokens, window n=128.

Query generator ("moving fixation"): at decode step t, for every layer and
query head h (served by KV head h // (H_q/H_kv)),
``q = g + 3 * mean(K rows of the 3x3 patch window centred at cell c_t)`` with
``g ~ N(0, 1)``; the window is clipped to the image grid (the mean runs over
the cells that exist) and ``c_t`` advances through the grid in raster order.
K and V are N(0, 1). R-SWA workloads use q ~ N(0, 1) instead.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import torch

__all__ = ["Workload", "WORKLOADS", "DecodeCase", "make_case", "workload"]


@dataclass(frozen=True)
class Workload:
    """Shape and schedule of one synthetic decode workload."""

    name: str
    batch: int
    layers: int
    q_heads: int
    kv_heads: int
    head_dim: int
    dtype: str                      # "f32" or "bf16": dtype of q, K, V and out
    prompt: int                     # text tokens before the image, positions [0, prompt)
    grid: tuple                     # (image pages, rows, cols); raster order, page-major
    steps: int                      # decode steps T (token t is at position prompt+N_img+t)
    tau: float = 1.0                # keep ratio of image tokens in focal layers
    warmup: int = 0                 # profiling warm-up steps w
    n_focal: int = 3                # |C| chosen by the profiler
    focal_layers: tuple | None = None   # fixed focal set (no profiling) when given
    page_size: int = 16             # tokens per KV page
    fixation: str = "raster"        # "raster" | "random_start"
    cells_per_step: int = 1         # fixation advance per decode step
    seed: int = 0
    mode: str = "fastocr"           # "fastocr" | "rswa"
    rswa_prefix: int = 0            # L_m (R-SWA global prefix length)
    rswa_window: int = 0            # n   (R-SWA window over generated tokens)
    extra: dict = field(default_factory=dict, compare=False)

    @property
    def n_img(self) -> int:
        pages, rows, cols = self.grid
        return pages * rows * cols

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def img_start(self) -> int:
        return self.prompt

    @property
    def max_tokens(self) -> int:
        """Cache length after the last decode step."""
        if self.mode == "rswa":
            return self.rswa_prefix + self.steps
        return self.prompt + self.n_img + self.steps

    def seq_len_at(self, t: int) -> int:
        """N_t: tokens in the cache at decode step t, the current token included."""
        if self.mode == "rswa":
            return self.rswa_prefix + t + 1
        return self.prompt + self.n_img + t + 1

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_f32": Workload(
        name="tiny_f32", batch=1, layers=2, q_heads=4, kv_heads=2, head_dim=64,
        dtype="f32", prompt=16, grid=(1, 16, 16), steps=32, tau=0.25, warmup=0,
        n_focal=1, focal_layers=(1,), seed=1),
    "qwen7b_b1": Workload(
        name="qwen7b_b1", batch=1, layers=28, q_heads=28, kv_heads=4, head_dim=128,
        dtype="bf16", prompt=64, grid=(1, 64, 64), steps=512, tau=0.05, warmup=8,
        n_focal=3, seed=2),
    "serving_b32": Workload(
        name="serving_b32", batch=32, layers=28, q_heads=28, kv_heads=4, head_dim=128,
        dtype="bf16", prompt=128, grid=(1, 128, 64), steps=256, tau=0.05, warmup=8,
        n_focal=3, fixation="random_start", seed=3),
    "multipage_b8": Workload(
        name="multipage_b8", batch=8, layers=28, q_heads=28, kv_heads=4, head_dim=128,
        dtype="bf16", prompt=64, grid=(4, 64, 64), steps=4096, tau=0.05, warmup=8,
        n_focal=3, cells_per_step=4, seed=4),
    "rswa_b16": Workload(
        name="rswa_b16", batch=16, layers=12, q_heads=10, kv_heads=10, head_dim=128,
        dtype="bf16", prompt=2624, grid=(1, 0, 0), steps=1024, mode="rswa",
        rswa_prefix=2560 + 64, rswa_window=128, seed=5),
}


def workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return w.with_(**overrides) if overrides else w


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


@dataclass
class DecodeCase:
    """Generated tensors of one workload, KV cache in paged layout.

    k_cache, v_cache: [layers, num_pages, H_kv, page_size, d]
    block_table:      [B, pages_per_seq] int32, page ids of sequence b in token order
    q:                [n_steps, layers, B, H_q, d] queries of decode steps
                      step0 .. step0+n_steps-1
    img_range:        [B, 2] int32 (start, length) of the image tokens
    """

    wl: Workload
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_table: torch.Tensor
    q: torch.Tensor
    img_range: torch.Tensor
    step0: int
    fixation_cells: torch.Tensor    # [n_steps, B] cell index of c_t (-1 for R-SWA)

    @property
    def device(self):
        return self.k_cache.device

    def seq_lens(self, t: int) -> torch.Tensor:
        return torch.full((self.wl.batch,), self.wl.seq_len_at(t), dtype=torch.int32,
                          device=self.device)

    def q_at(self, t: int) -> torch.Tensor:
        """[layers, B, H_q, d] queries of decode step t."""
        return self.q[t - self.step0]

    def logical_kv(self, layer: int, b: int, n_tokens: int):
        """K, V of sequence b in token order: two [n_tokens, H_kv, d] tensors."""
        return (_gather_logical(self.k_cache[layer], self.block_table[b], n_tokens),
                _gather_logical(self.v_cache[layer], self.block_table[b], n_tokens))


def _gather_logical(cache_l: torch.Tensor, bt_row: torch.Tensor, n_tokens: int) -> torch.Tensor:
    # cache_l: [num_pages, H_kv, page, d] -> [n_tokens, H_kv, d]
    page = cache_l.shape[2]
    n_pages = (n_tokens + page - 1) // page
    pages = cache_l[bt_row[:n_pages].long()]                  # [n_pages, H_kv, page, d]
    rows = pages.permute(0, 2, 1, 3).reshape(n_pages * page, cache_l.shape[1], cache_l.shape[3])
    return rows[:n_tokens]


def _generator(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def fixation_cells(wl: Workload, steps: range, gen_cpu: torch.Generator) -> torch.Tensor:
    """Cell index c_t (page-major raster) of each step and sequence: [len(steps), B]."""
    n_img = wl.n_img
    if wl.mode == "rswa" or n_img == 0:
        return torch.full((len(steps), wl.batch), -1, dtype=torch.int64)
    if wl.fixation == "random_start":
        start = torch.randint(0, n_img, (wl.batch,), generator=gen_cpu)
    else:
        start = torch.zeros(wl.batch, dtype=torch.int64)
    t = torch.tensor(list(steps), dtype=torch.int64)[:, None]
    return (start[None, :] + t * wl.cells_per_step) % n_img


def _window_offsets(wl: Workload, cells: torch.Tensor):
    """Image-token offsets of the 3x3 window around each cell, clipped to its page.

    cells: [S, B] -> (offsets [S, B, 9], valid [S, B, 9] bool)
    """
    pages, rows, cols = wl.grid
    per_page = rows * cols
    page = cells // per_page
    r = (cells % per_page) // cols
    c = cells % cols
    dr = torch.tensor([-1, -1, -1, 0, 0, 0, 1, 1, 1])
    dc = torch.tensor([-1, 0, 1, -1, 0, 1, -1, 0, 1])
    rr = r[..., None] + dr
    cc = c[..., None] + dc
    valid = (rr >= 0) & (rr < rows) & (cc >= 0) & (cc < cols)
    off = page[..., None] * per_page + rr.clamp(0, rows - 1) * cols + cc.clamp(0, cols - 1)
    return off, valid


def make_case(wl: Workload, device="cpu", step0: int = 0, n_steps: int | None = None,
              seed: int | None = None) -> DecodeCase:
    """Draw the KV cache (room for all wl.steps tokens) and the queries of steps
    [step0, step0 + n_steps). Same seed and device => same bytes."""
    device = torch.device(device)
    seed = wl.seed if seed is None else seed
    if n_steps is None:
        n_steps = wl.steps - step0
    dt = torch_dtype(wl.dtype)
    gen_cpu = _generator("cpu", seed)
    gen_dev = gen_cpu if device.type == "cpu" else _generator(device, seed + 7919)

    ps = wl.page_size
    pages_per_seq = (wl.max_tokens + ps - 1) // ps
    num_pages = wl.batch * pages_per_seq
    # pages handed out in a seeded random order, so no sequence is contiguous
    perm = torch.randperm(num_pages, generator=gen_cpu).to(torch.int32)
    block_table = perm.view(wl.batch, pages_per_seq).contiguous()

    shape = (wl.layers, num_pages, wl.kv_heads, ps, wl.head_dim)
    k_cache = torch.randn(shape, generator=gen_dev, device=device, dtype=torch.float32).to(dt)
    v_cache = torch.randn(shape, generator=gen_dev, device=device, dtype=torch.float32).to(dt)

    steps = range(step0, step0 + n_steps)
    cells = fixation_cells(wl, steps, gen_cpu)
    qshape = (n_steps, wl.layers, wl.batch, wl.q_heads, wl.head_dim)
    q = torch.empty(qshape, device=device, dtype=dt)
    chunk = 32
    for s0 in range(0, n_steps, chunk):
        s1 = min(n_steps, s0 + chunk)
        g = torch.randn((s1 - s0,) + qshape[1:], generator=gen_dev, device=device,
                        dtype=torch.float32)
        if wl.mode == "rswa" or wl.n_img == 0:
            q[s0:s1] = g.to(dt)
        else:
            q[s0:s1] = (g + 3.0 * _window_mean(wl, k_cache, block_table, cells[s0:s1])).to(dt)

    img = torch.tensor([[wl.img_start, wl.n_img]] * wl.batch, dtype=torch.int32)
    return DecodeCase(wl=wl, k_cache=k_cache, v_cache=v_cache,
                      block_table=block_table.to(device), q=q, img_range=img.to(device),
                      step0=step0, fixation_cells=cells)


def _window_mean(wl: Workload, k_cache, block_table, cells) -> torch.Tensor:
    """mean of K over the clipped 3x3 window: [S, L, B, H_q, d] (fp32)."""
    off, valid = _window_offsets(wl, cells)                     # [S, B, 9]
    pos = wl.img_start + off                                    # cache positions
    ps = wl.page_size
    bt = block_table.to(k_cache.device).long()
    b_idx = torch.arange(wl.batch)[None, :, None].expand_as(pos)
    page = bt[b_idx.to(bt.device), (pos // ps).to(bt.device)]   # [S, B, 9]
    slot = (pos % ps).to(k_cache.device)
    # [L, P, H, ps, d] -> [P, ps, L, H, d], then rows of the windows: [S, B, 9, L, H, d]
    rows = k_cache.permute(1, 3, 0, 2, 4)[page, slot].float()
    w = valid.to(k_cache.device).float()[:, :, :, None, None, None]
    mean = (rows * w).sum(2) / w.sum(2)                          # [S, B, L, H_kv, d]
    mean = mean.permute(0, 2, 1, 3, 4)                           # [S, L, B, H_kv, d]
    return mean.repeat_interleave(wl.group, dim=3)              # [S, L, B, H_q, d]
