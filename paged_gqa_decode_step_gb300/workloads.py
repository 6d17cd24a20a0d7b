"""Seeded synthetic inputs for the paged decode step.

This module only draws random numbers and lays out page tables; it holds none
of the method's arithmetic, so that the CPU oracle and the CUDA path can both
be fed from it without sharing any computation.

The shapes follow the model pages:
  * llama-3.1-8b-instruct architecture page, "Generics" (H 4096, Heads 32,
    KvHeads 8, MaxSeq 8192) and GroupedQueryAttention (PageSize 64);
  * gpt-oss-20b architecture page, "Generics" (Heads 64, KvHeads 8, HeadDim 64,
    Window 128, MaxSeq 4096);
  * gpt2 architecture page, "Generics" (H 768, Heads 12, MaxSeq 1024, T f32).

Recipe (every workload): draws come from one ``torch.Generator`` seeded with
the workload's seed, in the order positions -> page permutation -> q -> k_new
-> v_new -> k_pool -> v_pool.  Values are N(0, 1) drawn in f32 and rounded to
the element type.  The pool holds sum_r ceil((pos_r + 1) / 64) pages plus 10%
spare (or an explicit count); page ids are a seeded permutation of the pool,
handed to rows in row order, and table entries past a row's last page are -1.
The prefilled pool stands for keys that were rotated when they were written.
"""
from dataclasses import dataclass, field, replace
import math
from typing import Optional, Sequence

import torch

PAGE_SIZE = 64


@dataclass(frozen=True)
class Workload:
    name: str
    rows: int
    heads: int
    kv_heads: int
    head_dim: int
    pages_per_row: int
    dtype: str                      # "bf16" or "f32"
    rope_theta: float               # <= 0: no rotation
    window: int = 0                 # <= 0: attend every position up to pos
    positions: str = "uniform"      # "fixed" | "uniform" | "loguniform_ctx"
    pos_lo: int = 0
    pos_hi: int = 0
    fixed_positions: Sequence[int] = field(default_factory=tuple)
    num_pages: int = 0              # 0: needed pages + 10% spare
    seed: int = 0

    @property
    def group(self) -> int:
        return self.heads // self.kv_heads

    @property
    def max_seq(self) -> int:
        return self.pages_per_row * PAGE_SIZE

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4


# The five workloads, in the order they are listed for this step.
TINY = Workload("tiny", rows=2, heads=8, kv_heads=8, head_dim=64, pages_per_row=8, dtype="bf16",
                rope_theta=10000.0, positions="fixed", fixed_positions=(37, 100), num_pages=16,
                seed=1000)
LLAMA_LAYER = Workload("llama8b_layer", rows=32, heads=32, kv_heads=8, head_dim=128,
                       pages_per_row=128, dtype="bf16", rope_theta=500000.0, positions="uniform",
                       pos_lo=1024, pos_hi=8191, seed=1001)
LLAMA_SERVING = Workload("llama8b_serving", rows=256, heads=32, kv_heads=8, head_dim=128,
                         pages_per_row=128, dtype="bf16", rope_theta=500000.0,
                         positions="loguniform_ctx", pos_lo=16, pos_hi=8192, seed=1002)
GPTOSS_FULL = Workload("gptoss20b_full", rows=64, heads=64, kv_heads=8, head_dim=64,
                       pages_per_row=64, dtype="bf16", rope_theta=150000.0, window=0,
                       positions="uniform", pos_lo=256, pos_hi=4095, seed=1003)
GPTOSS_SLIDING = replace(GPTOSS_FULL, name="gptoss20b_sliding", window=128)
GPT2 = Workload("gpt2_f32", rows=128, heads=12, kv_heads=12, head_dim=64, pages_per_row=16,
                dtype="f32", rope_theta=0.0, positions="uniform", pos_lo=1, pos_hi=1023,
                seed=1004)

WORKLOADS = {w.name: w for w in (TINY, LLAMA_LAYER, LLAMA_SERVING, GPTOSS_FULL, GPTOSS_SLIDING, GPT2)}


def draw_positions(w: Workload, gen: torch.Generator) -> torch.Tensor:
    """Positions [rows] int32 on the generator's device."""
    dev = gen.device
    if w.positions == "fixed":
        assert len(w.fixed_positions) == w.rows
        return torch.tensor(list(w.fixed_positions), dtype=torch.int32, device=dev)
    if w.positions == "uniform":
        return torch.randint(w.pos_lo, w.pos_hi + 1, (w.rows,), generator=gen, device=dev,
                             dtype=torch.int64).to(torch.int32)
    if w.positions == "loguniform_ctx":
        u = torch.rand((w.rows,), generator=gen, device=dev, dtype=torch.float64)
        lo, hi = math.log(w.pos_lo), math.log(w.pos_hi)
        ctx = torch.floor(torch.exp(lo + (hi - lo) * u)).clamp(w.pos_lo, w.pos_hi)
        return (ctx - 1).to(torch.int32)
    raise ValueError(w.positions)


def pages_needed(positions: torch.Tensor) -> torch.Tensor:
    """Pages each row owns: ceil((pos + 1) / 64)."""
    return (positions.to(torch.int64) + PAGE_SIZE) // PAGE_SIZE


def generate(w: Workload, device="cpu", seed: Optional[int] = None, poison: bool = False):
    """Draw one step's inputs.

    Returns a dict of tensors on ``device``: q [R, Hq, D], k_new / v_new
    [R, Hk, D], positions [R] i32, table [R, Pages] i32, k_pool / v_pool
    [NumPages, Hk, 64, D].  With ``poison``, pool slots that no row may read
    (spare pages, slots past a row's position in its last page and slots
    before its window) hold NaN, so that any read of them shows in the output.
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    positions = draw_positions(w, gen)
    assert int(positions.max()) < w.max_seq and int(positions.min()) >= 0
    need = pages_needed(positions)
    total = int(need.sum())
    num_pages = w.num_pages if w.num_pages > 0 else total + math.ceil(total * 0.1)
    assert num_pages >= total
    perm = torch.randperm(num_pages, generator=gen, device=device).to(torch.int32)
    table = torch.full((w.rows, w.pages_per_row), -1, dtype=torch.int32, device=device)
    need_cpu = need.cpu().tolist()
    off = 0
    for r, n in enumerate(need_cpu):
        table[r, :n] = perm[off:off + n]
        off += n

    def normal(*shape):
        return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32).to(w.torch_dtype)

    R, Hq, Hk, D = w.rows, w.heads, w.kv_heads, w.head_dim
    q = normal(R, Hq, D)
    k_new = normal(R, Hk, D)
    v_new = normal(R, Hk, D)
    k_pool = normal(num_pages, Hk, PAGE_SIZE, D)
    v_pool = normal(num_pages, Hk, PAGE_SIZE, D)
    if poison:
        _poison(w, positions, table, k_pool, v_pool)
    return dict(q=q, k_new=k_new, v_new=v_new, positions=positions, table=table,
                k_pool=k_pool, v_pool=v_pool)


def _poison(w, positions, table, k_pool, v_pool):
    nan = float("nan")
    used = torch.zeros(k_pool.shape[0], dtype=torch.bool, device=k_pool.device)
    pos_cpu = positions.cpu().tolist()
    tab_cpu = table.cpu()
    for r, pos in enumerate(pos_cpu):
        lo = max(0, pos - w.window + 1) if w.window > 0 else 0
        n = pos // PAGE_SIZE + 1
        pages = tab_cpu[r, :n].tolist()
        used[torch.tensor(pages, dtype=torch.int64, device=k_pool.device)] = True
        last = pages[-1]
        k_pool[last, :, pos % PAGE_SIZE + 1:, :] = nan
        v_pool[last, :, pos % PAGE_SIZE + 1:, :] = nan
        for t_page in range(lo // PAGE_SIZE):
            k_pool[pages[t_page]] = nan
            v_pool[pages[t_page]] = nan
        if lo % PAGE_SIZE:
            first = pages[lo // PAGE_SIZE]
            k_pool[first, :, :lo % PAGE_SIZE, :] = nan
            v_pool[first, :, :lo % PAGE_SIZE, :] = nan
    k_pool[~used] = nan
    v_pool[~used] = nan


def to_numpy(t: torch.Tensor):
    """Host numpy view for the oracle: bf16 as uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()


def from_numpy(a, dtype) -> torch.Tensor:
    """Inverse of to_numpy."""
    t = torch.from_numpy(a.copy())
    if dtype == torch.bfloat16:
        return t.view(torch.int16).view(torch.bfloat16)
    return t


@dataclass(frozen=True)
class PrefillWorkload:
    """Packed prompt chunks: row r holds `prefix[r]` cached positions and gets
    `chunk[r]` new tokens at positions prefix[r] .. prefix[r] + chunk[r] - 1,
    packed row after row."""
    name: str
    prefix: Sequence[int]
    chunk: Sequence[int]
    heads: int
    kv_heads: int
    head_dim: int
    pages_per_row: int
    dtype: str = "bf16"
    rope_theta: float = 10000.0
    window: int = 0
    seed: int = 0

    @property
    def rows(self) -> int:
        return len(self.prefix)

    @property
    def tokens(self) -> int:
        return int(sum(self.chunk))

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def max_seq(self) -> int:
        return self.pages_per_row * PAGE_SIZE


def generate_prefill(w: PrefillWorkload, device="cpu", seed: Optional[int] = None):
    """Inputs of one prefill call: q [P, Hq, D], k_new / v_new [P, Hk, D],
    positions / rows / slots [P] i32 (slot = page * 64 + offset of the token's
    position in its row), table [R, Pages] i32, pools [NumPages, Hk, 64, D].
    Draw order: page permutation -> q -> k_new -> v_new -> k_pool -> v_pool;
    the pool is N(0, 1) everywhere, so every prefix position holds a key."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    ends = [p + c for p, c in zip(w.prefix, w.chunk)]
    assert max(ends) <= w.max_seq
    need = [(e + PAGE_SIZE - 1) // PAGE_SIZE for e in ends]
    total = sum(need)
    num_pages = total + math.ceil(total * 0.1)
    perm = torch.randperm(num_pages, generator=gen, device=device).to(torch.int32).cpu()
    table = torch.full((w.rows, w.pages_per_row), -1, dtype=torch.int32)
    off = 0
    for r, n in enumerate(need):
        table[r, :n] = perm[off:off + n]
        off += n
    positions, rows, slots = [], [], []
    for r, (p0, c) in enumerate(zip(w.prefix, w.chunk)):
        for t in range(p0, p0 + c):
            positions.append(t)
            rows.append(r)
            slots.append(int(table[r, t // PAGE_SIZE]) * PAGE_SIZE + t % PAGE_SIZE)

    def normal(*shape):
        return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32).to(w.torch_dtype)

    P, Hq, Hk, D = w.tokens, w.heads, w.kv_heads, w.head_dim
    i32 = lambda x: torch.tensor(x, dtype=torch.int32, device=device)
    return dict(q=normal(P, Hq, D), k_new=normal(P, Hk, D), v_new=normal(P, Hk, D), positions=i32(positions),
                rows=i32(rows), slots=i32(slots), table=table.to(device),
                k_pool=normal(num_pages, Hk, PAGE_SIZE, D), v_pool=normal(num_pages, Hk, PAGE_SIZE, D))


# Llama-3.1-8B attention shape, chunked prefill: 8 rows, 1024 new tokens each
# on cached prefixes of 0, 1024, ..., 7168 positions (8192 tokens in all,
# contexts 1 .. 8192).
PREFILL_LLAMA = PrefillWorkload("llama8b_prefill", prefix=tuple(range(0, 8192, 1024)), chunk=(1024,) * 8,
                                heads=32, kv_heads=8, head_dim=128, pages_per_row=128, rope_theta=500000.0,
                                seed=1005)

PREFILL_WORKLOADS = {w.name: w for w in (PREFILL_LLAMA,)}


@dataclass(frozen=True)
class PackedWorkload:
    """Sequences of the given lengths packed into one row: sequence s holds
    positions 0 .. lengths[s] - 1; its segment id is s, or a shuffled id."""
    name: str
    lengths: Sequence[int]
    heads: int
    kv_heads: int
    head_dim: int
    dtype: str = "bf16"
    rope_theta: float = 10000.0
    window: int = 0
    shuffle_ids: bool = False
    seed: int = 0

    @property
    def tokens(self) -> int:
        return int(sum(self.lengths))

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def max_seq(self) -> int:
        return int(max(self.lengths))


def generate_packed(w: PackedWorkload, device="cpu", seed: Optional[int] = None):
    """q [P, Hq, D], k / v [P, Hk, D], positions / segments [P] i32.
    Draw order: segment ids (if shuffled) -> q -> k -> v."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    n_seq = len(w.lengths)
    ids = torch.randperm(n_seq, generator=gen, device=device).cpu().tolist() if w.shuffle_ids else list(range(n_seq))
    positions, segments = [], []
    for s, L in enumerate(w.lengths):
        positions += list(range(L))
        segments += [ids[s] * 7 + 3] * L          # arbitrary, non-contiguous id values
    P, Hq, Hk, D = w.tokens, w.heads, w.kv_heads, w.head_dim

    def normal(*shape):
        return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32).to(w.torch_dtype)

    i32 = lambda x: torch.tensor(x, dtype=torch.int32, device=device)
    return dict(q=normal(P, Hq, D), k=normal(P, Hk, D), v=normal(P, Hk, D), positions=i32(positions),
                segments=i32(segments))


# Llama-3.1-8B attention shape, packed training row: 8192 tokens in sequences
# of mixed lengths (the pages' packed entries take several sequences per row).
PACKED_LLAMA = PackedWorkload("llama8b_packed", lengths=(3000, 1500, 1200, 900, 700, 400, 300, 192), heads=32,
                              kv_heads=8, head_dim=128, rope_theta=500000.0, seed=1006)

PACKED_WORKLOADS = {w.name: w for w in (PACKED_LLAMA,)}
