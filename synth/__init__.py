"""Seeded synthetic inputs for the LOCKS decode step.

This module is shared by the CUDA path's tests/benchmark and by the float64
oracle. It only draws random numbers and lays them out; it holds none of the
method's arithmetic (no summary build, no scoring, no selection, no attention).

Shapes and value distributions follow the workloads described on the LOCKS
pages ("How LOCKS works" on the wps.hkprog.org post: page of 16 keys,
d_head = 128, rank 8) and the five decode configurations this project is
measured on:

* page-local low-rank keys  K_j = mu_j + A_j B_j + 0.05 N(0, 1)
  with mu_j ~ N(0, 0.5^2)^128, B_j an 8 x 128 matrix with orthonormal rows
  (QR of a Gaussian, sign fixed by diag(R)) and A_j ~ N(0, 1)^(16 x 8);
* rank-4 pages (same with 4 in place of 8) and isotropic N(0, 1) pages;
* carrier pages whose centroid has cosine 0.8 with the group's query
  direction: mu_j = |mu'| (0.8 q_hat + 0.6 u_perp);
* values V ~ N(0, 1), queries q ~ N(0, 1) in fp32; K and V rounded to bf16
  (round to nearest even) as the configurations state.

Layouts (all C-contiguous numpy arrays):

* ``k_cache`` / ``v_cache``: uint16 bf16 bits ``[num_phys_pages][Hkv][16][128]``
* ``q``: float32 ``[B][Hq][128]``; query head h belongs to kv head h // g
* ``page_table``: int32 ``[B][max_pages]`` logical page -> physical page
* ``seq_pages``: int32 ``[B]`` number of full pages of each sequence

Every stream is derived from ``numpy.random.SeedSequence(seed, spawn_key=...)``
with a fixed key per purpose and chunk, so a chunk can be regenerated on its
own and the output does not depend on the machine.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

PAGE = 16
D_HEAD = 128
RANK = 8
CHUNK_PAGES = 2048  # pages generated per random stream

# purposes used in the spawn keys
_KEYS, _VALUES, _QUERY, _CARRIER, _TYPES, _TABLE, _SUMMARY = range(7)

PAGE_LOWRANK8, PAGE_LOWRANK4, PAGE_ISO = 0, 1, 2


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode configuration (sizes, mix, seeds)."""

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    pages: int  # full pages per sequence
    budgets: Tuple[int, ...]
    carriers_per_kv_head: int
    seeds: Tuple[int, ...]  # one per request, or a single seed for all
    shuffled_table: bool = False
    type_mix: Tuple[float, float, float] = (1.0, 0.0, 0.0)  # lowrank8, lowrank4, iso
    description: str = ""

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def context(self) -> int:
        return self.pages * PAGE

    @property
    def num_phys_pages(self) -> int:
        return self.batch * self.pages

    def seed_of(self, b: int) -> int:
        return self.seeds[b] if len(self.seeds) > 1 else self.seeds[0]

    def scaled(self, pages: Optional[int] = None, batch: Optional[int] = None,
               name_suffix: str = "-small") -> "Workload":
        """Same shapes and mix with fewer pages / requests (for quick tests)."""
        p = self.pages if pages is None else pages
        b = self.batch if batch is None else batch
        seeds = self.seeds if len(self.seeds) == 1 else self.seeds[:b]
        carriers = min(self.carriers_per_kv_head, max(1, p // 8))
        return dataclasses.replace(self, name=self.name + name_suffix, pages=p, batch=b,
                                   seeds=seeds, carriers_per_kv_head=carriers)


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 1, 1, 1, 256, (256,), 4, (0,),
                     description="tiny single-head instance, 4K context, budget 256"),
    "llama8b_128k": Workload("llama8b_128k", 1, 32, 8, 8192, (2048,), 16, (1,),
                             description="Llama-3.1-8B-shaped layer, 128K context, budget 2048"),
    "batch8_256k": Workload("batch8_256k", 8, 32, 8, 16384, (512, 2048), 16,
                            tuple(range(2, 10)), shuffled_table=True,
                            description="8 requests x 256K, shuffled page table, budgets 512/2048"),
    "ctx1m": Workload("ctx1m", 1, 32, 8, 65536, (512, 2048), 32, (10,),
                      type_mix=(0.7, 0.2, 0.1),
                      description="1M context, 70/20/10 rank-8/rank-4/isotropic pages"),
    "glm9b_4x1m": Workload("glm9b_4x1m", 4, 32, 2, 65536, (512,), 16, (11,),
                           description="GLM-4-9B-shaped, 4 x 1M, GQA group 16, budget 512"),
}


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(seed, spawn_key=tuple(int(k) for k in key)))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    nan = np.isnan(x)
    out = rounded.astype(np.uint16)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def make_query(w: Workload, b: int) -> np.ndarray:
    """q ~ N(0, 1) in fp32, [Hq][128] for request b."""
    return _rng(w.seed_of(b), _QUERY, b).standard_normal((w.num_q_heads, D_HEAD), dtype=np.float32)


def make_queries(w: Workload) -> np.ndarray:
    return np.stack([make_query(w, b) for b in range(w.batch)]).astype(np.float32)


def page_types(w: Workload, b: int, kvh: int) -> np.ndarray:
    """Per-page type for (request, kv head): a seeded shuffle of the configured mix."""
    n8 = int(round(w.type_mix[0] * w.pages))
    n4 = int(round(w.type_mix[1] * w.pages))
    n4 = min(n4, w.pages - n8)
    types = np.full(w.pages, PAGE_ISO, dtype=np.int8)
    types[:n8] = PAGE_LOWRANK8
    types[n8:n8 + n4] = PAGE_LOWRANK4
    if w.type_mix != (1.0, 0.0, 0.0):
        _rng(w.seed_of(b), _TYPES, b, kvh).shuffle(types)
    return types


def carrier_pages(w: Workload, b: int, kvh: int, q: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Distinct carrier page ids and their centroids for (request, kv head).

    The query direction of a kv head is the normalised sum of its group's query
    heads. Each carrier centroid has cosine 0.8 with it and the norm of a fresh
    N(0, 0.5^2) draw.
    """
    g = w.group
    n = min(w.carriers_per_kv_head, w.pages)
    rng = _rng(w.seed_of(b), _CARRIER, b, kvh)
    pages = np.sort(rng.choice(w.pages, size=n, replace=False)).astype(np.int64)
    qsum = q[kvh * g:(kvh + 1) * g].astype(np.float64).sum(axis=0)
    qhat = qsum / np.linalg.norm(qsum)
    mus = np.empty((n, D_HEAD), dtype=np.float64)
    for i in range(n):
        mu_prime = 0.5 * rng.standard_normal(D_HEAD)
        u = rng.standard_normal(D_HEAD)
        u -= (u @ qhat) * qhat
        u /= np.linalg.norm(u)
        mus[i] = np.linalg.norm(mu_prime) * (0.8 * qhat + 0.6 * u)
    return pages, mus


def _orthonormal_rows(rng: np.random.Generator, n: int, r: int) -> np.ndarray:
    """n random r x 128 matrices with orthonormal rows (QR of a Gaussian, sign by diag(R))."""
    g = rng.standard_normal((n, D_HEAD, r))
    qm, rm = np.linalg.qr(g)
    sign = np.sign(np.diagonal(rm, axis1=1, axis2=2))
    sign[sign == 0] = 1.0
    qm = qm * sign[:, None, :]
    return np.transpose(qm, (0, 2, 1))  # (n, r, 128)


def make_keys_chunk(w: Workload, b: int, kvh: int, p0: int, p1: int,
                    types: np.ndarray, carriers: Tuple[np.ndarray, np.ndarray]) -> np.ndarray:
    """fp32 keys of logical pages [p0, p1) for (request, kv head): (n, 16, 128)."""
    n = p1 - p0
    rng = _rng(w.seed_of(b), _KEYS, b, kvh, p0 // CHUNK_PAGES)
    t = types[p0:p1]
    mu = 0.5 * rng.standard_normal((n, D_HEAD))
    noise = rng.standard_normal((n, PAGE, D_HEAD), dtype=np.float32)
    keys = np.empty((n, PAGE, D_HEAD), dtype=np.float64)
    for rank, ptype in ((8, PAGE_LOWRANK8), (4, PAGE_LOWRANK4)):
        idx = np.nonzero(t == ptype)[0]
        if idx.size == 0:
            continue
        basis = _orthonormal_rows(rng, idx.size, rank)
        coeff = rng.standard_normal((idx.size, PAGE, rank))
        keys[idx] = mu[idx, None, :] + np.matmul(coeff, basis) + 0.05 * noise[idx]
    iso = np.nonzero(t == PAGE_ISO)[0]
    if iso.size:
        keys[iso] = noise[iso]
    cpages, cmus = carriers
    sel = (cpages >= p0) & (cpages < p1)
    for cp, cmu in zip(cpages[sel], cmus[sel]):
        j = int(cp - p0)
        own_mu = mu[j] if t[j] != PAGE_ISO else 0.0
        keys[j] = keys[j] - own_mu + cmu[None, :]
    return keys.astype(np.float32)


def make_values_chunk(w: Workload, b: int, kvh: int, p0: int, p1: int) -> np.ndarray:
    rng = _rng(w.seed_of(b), _VALUES, b, kvh, p0 // CHUNK_PAGES)
    return rng.standard_normal((p1 - p0, PAGE, D_HEAD), dtype=np.float32)


def make_page_table(w: Workload) -> np.ndarray:
    """[B][P] logical -> physical page. Identity blocks, or a seeded permutation of the pool."""
    ids = np.arange(w.num_phys_pages, dtype=np.int64)
    if w.shuffled_table:
        _rng(w.seeds[0], _TABLE).shuffle(ids)
    return ids.reshape(w.batch, w.pages).astype(np.int32)


@dataclasses.dataclass
class DecodeInputs:
    workload: Workload
    q: np.ndarray            # float32 [B][Hq][128]
    k_cache: np.ndarray      # uint16 (bf16) [num_phys][Hkv][16][128]
    v_cache: np.ndarray      # uint16 (bf16) [num_phys][Hkv][16][128]
    page_table: np.ndarray   # int32 [B][P]
    seq_pages: np.ndarray    # int32 [B]
    carriers: List[List[np.ndarray]]  # [b][kvh] -> sorted carrier logical page ids
    types: List[List[np.ndarray]]     # [b][kvh] -> page types


def _fill_chunk(w: Workload, b: int, kvh: int, p0: int, k_cache: np.ndarray, v_cache: Optional[np.ndarray],
                table: np.ndarray, q: np.ndarray) -> None:
    p1 = min(w.pages, p0 + CHUNK_PAGES)
    types = page_types(w, b, kvh)
    car = carrier_pages(w, b, kvh, q[b])
    phys = table[b, p0:p1]
    k_cache[phys, kvh] = f32_to_bf16_bits(make_keys_chunk(w, b, kvh, p0, p1, types, car))
    if v_cache is not None:
        v_cache[phys, kvh] = f32_to_bf16_bits(make_values_chunk(w, b, kvh, p0, p1))


def _chunk_task(args) -> None:
    """Worker body: attach to the shared K/V buffers and fill one (b, kv head, chunk)."""
    from multiprocessing import shared_memory
    w, b, kvh, p0, k_name, v_name, shape = args
    shm_k = shared_memory.SharedMemory(name=k_name)
    shm_v = shared_memory.SharedMemory(name=v_name) if v_name else None
    try:
        k = np.ndarray(shape, dtype=np.uint16, buffer=shm_k.buf)
        v = np.ndarray(shape, dtype=np.uint16, buffer=shm_v.buf) if shm_v else None
        _fill_chunk(w, b, kvh, p0, k, v, make_page_table(w), make_queries(w))
        del k, v
    finally:
        shm_k.close()
        if shm_v:
            shm_v.close()


def make_decode_inputs(w: Workload, with_values: bool = True, workers: int = 0) -> DecodeInputs:
    """Generate the full paged K/V cache, queries and page table of a workload.

    Each (request, kv head, chunk of pages) has its own random stream, so the
    result does not depend on ``workers``; with workers > 1 the chunks are
    generated by a spawn-started process pool writing into shared memory.
    """
    q = make_queries(w)
    table = make_page_table(w)
    shape = (w.num_phys_pages, w.num_kv_heads, PAGE, D_HEAD)
    tasks = [(b, kvh, p0) for b in range(w.batch) for kvh in range(w.num_kv_heads)
             for p0 in range(0, w.pages, CHUNK_PAGES)]
    if workers > 1 and len(tasks) > 1:
        import multiprocessing as mp
        from multiprocessing import shared_memory
        nbytes = int(np.prod(shape)) * 2
        shm_k = shared_memory.SharedMemory(create=True, size=nbytes)
        shm_v = shared_memory.SharedMemory(create=True, size=nbytes) if with_values else None
        try:
            args = [(w, b, kvh, p0, shm_k.name, shm_v.name if shm_v else None, shape) for b, kvh, p0 in tasks]
            from concurrent.futures import ProcessPoolExecutor
            # spawn (not fork: callers may already hold a CUDA context); a worker
            # that dies raises BrokenProcessPool instead of being respawned
            with ProcessPoolExecutor(min(workers, len(tasks)), mp_context=mp.get_context("spawn")) as ex:
                list(ex.map(_chunk_task, args))
            k_cache = np.ndarray(shape, dtype=np.uint16, buffer=shm_k.buf).copy()
            v_cache = (np.ndarray(shape, dtype=np.uint16, buffer=shm_v.buf).copy() if shm_v
                       else np.zeros((0,), np.uint16))
        finally:
            shm_k.close()
            shm_k.unlink()
            if shm_v:
                shm_v.close()
                shm_v.unlink()
    else:
        k_cache = np.empty(shape, dtype=np.uint16)
        v_cache = np.empty(shape, dtype=np.uint16) if with_values else np.zeros((0,), np.uint16)
        for b, kvh, p0 in tasks:
            _fill_chunk(w, b, kvh, p0, k_cache, v_cache if with_values else None, table, q)
    carriers = [[carrier_pages(w, b, kvh, q[b])[0] for kvh in range(w.num_kv_heads)] for b in range(w.batch)]
    types_all = [[page_types(w, b, kvh) for kvh in range(w.num_kv_heads)] for b in range(w.batch)]
    seq_pages = np.full(w.batch, w.pages, dtype=np.int32)
    return DecodeInputs(w, q, k_cache, v_cache, table, seq_pages, carriers, types_all)


@dataclasses.dataclass
class SummaryBytes:
    """Raw summary arrays in the library's layout (codes and fp16 scale bits)."""

    mu: np.ndarray      # int8  [num_phys][Hkv][128]
    basis: np.ndarray   # uint8 [num_phys][Hkv][512]  (two int4 codes per byte)
    coef: np.ndarray    # int8  [num_phys][Hkv][128]
    scales: np.ndarray  # uint16 [num_phys][Hkv][4]  fp16 bits (mu, basis, coef, 0)


def _f16_bits(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def random_summaries(num_phys: int, num_kv_heads: int, seed: int,
                     extreme_fraction: float = 0.0) -> SummaryBytes:
    """Random, valid summary bytes (any code in range, positive fp16 scales).

    Used to drive the scorer at full size without a build: codes are uniform
    over [-127, 127] (int8 arrays) and [-7, 7] (int4 basis; the nibble 0b1000
    is never produced), scales are positive fp16 values of the magnitudes a
    build of the generator's keys gives. ``extreme_fraction`` of the units get
    all-extreme codes (+-127 / +-7) to exercise the largest products.
    """
    rng = _rng(seed, _SUMMARY)
    n = num_phys * num_kv_heads
    mu = rng.integers(-127, 128, size=(n, 128), dtype=np.int16).astype(np.int8)
    coef = rng.integers(-127, 128, size=(n, 128), dtype=np.int16).astype(np.int8)
    nib = rng.integers(0, 15, size=(n, 1024), dtype=np.int16)  # 0..14
    nib = np.where(nib >= 8, nib + 1, nib).astype(np.uint8)     # skip 8 (= -8)
    if extreme_fraction > 0:
        m = rng.random(n) < extreme_fraction
        k = int(m.sum())
        if k:
            sgn = rng.integers(0, 2, size=(k, 128)) * 2 - 1
            mu[m] = (127 * sgn).astype(np.int8)
            sgn = rng.integers(0, 2, size=(k, 128)) * 2 - 1
            coef[m] = (127 * sgn).astype(np.int8)
            sgn = rng.integers(0, 2, size=(k, 1024))
            nib[m] = np.where(sgn == 1, 7, 9).astype(np.uint8)  # +7 or -7
    basis = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    s_mu = rng.uniform(1.0, 3.0, n) / 127.0
    s_v = rng.uniform(0.2, 0.5, n) / 7.0
    s_c = rng.uniform(2.0, 5.0, n) / 127.0
    scales = np.zeros((n, 4), dtype=np.uint16)
    scales[:, 0] = _f16_bits(s_mu)
    scales[:, 1] = _f16_bits(s_v)
    scales[:, 2] = _f16_bits(s_c)
    return SummaryBytes(mu.reshape(num_phys, num_kv_heads, 128),
                        basis.reshape(num_phys, num_kv_heads, 512),
                        coef.reshape(num_phys, num_kv_heads, 128),
                        scales.reshape(num_phys, num_kv_heads, 4))


def random_cache(num_phys: int, num_kv_heads: int, seed: int, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) bf16 page pool [num_phys][Hkv][16][128] (no page structure)."""
    rng = _rng(seed, _VALUES, 1 << 20)
    x = std * rng.standard_normal((num_phys, num_kv_heads, PAGE, D_HEAD), dtype=np.float32)
    return f32_to_bf16_bits(x)


def ragged_seq_pages(batch: int, max_pages: int, seed: int, min_pages: int = 0) -> np.ndarray:
    rng = _rng(seed, _TABLE, 7)
    return rng.integers(min_pages, max_pages + 1, size=batch).astype(np.int32)
