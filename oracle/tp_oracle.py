"""fp64 CPU oracle of the Megatron tensor-parallel layers (test infrastructure).

Every function restates one passage of the pages on tensor parallelism in
plain numpy, in float64, with no blocking, fusion or reordering beyond what
the passage states.  A numpy matmul is used as a library step where a
passage multiplies matrices.  Nothing in this module is imported by the
CUDA library; only tests, ``smoke()`` and the CPU legs of ``bench.py`` use it.

Page titles used in the citations below:

* "vLLM source analysis 13: tensor parallelism in detail" (171host.com):
  §1.1.1 Reduce-Scatter, §1.1.2 All-Gather, §1.2 ring cost, low-latency
  all-reduce pseudocode after §1.2, §2.2 MLP, §2.4.1 input embedding,
  §2.4.2 output embedding.
* "Nano-vLLM walkthrough 22: tensor parallelism (2), code" (mokono.cn):
  §3 ColumnParallelLinear, §4 RowParallelLinear, §5 merged double cut.
* "Tensor parallelism from scratch" (AI-infra handbook): tp.py listing
  (VocabParallelEmbedding, TPMLP, TPTransformer), "the cost of communication".
* "6.2 Tensor-parallel inference" (AIInfraGuide): §1 FFN formula
  Y = sum_i act(X A_i) B_i, §3.1 all-reduce time.
* "Mini-SGLang source reading: TP": §2-§5 column/row/vocab recap.

Readings where the pages are silent are listed next to the function that
takes them.
"""

from __future__ import annotations

import math
from typing import Dict, List, Sequence, Tuple

import numpy as np

__all__ = [
    "bf16_bits_to_f64", "f32_bits_to_f64", "round_to_bf16", "bf16_from_f64_bits",
    "divide", "column_shard", "row_shard", "merged_column_shard", "qkv_shard", "qkv_shard_gqa", "kv_head_of_rank",
    "vocab_range", "linear", "silu", "gelu_tanh", "glu",
    "mlp_unsharded", "mlp_shard_partials", "mlp_sharded", "round_to_f32", "mlp_sharded_rounded",
    "reduce_direct", "reduce_direct_f32", "ring_chunks", "ring_schedule",
    "ring_allreduce", "ring_fold_order",
    "vocab_parallel_embedding", "lm_head_sharded", "lm_head_unsharded", "shard_gather",
    "allreduce_time",
    "rmsnorm", "token_chunks", "ring_reduce_scatter", "reduce_scatter_fold_order",
    "all_gather_rows", "sequence_parallel_residual_norm",
]


# ---------------------------------------------------------------------------
# Number formats.  The oracle reads the exact bit patterns the GPU gets and
# widens them exactly to float64.
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bfloat16 bit patterns (uint16) as float64.

    bfloat16 is the top half of an IEEE binary32, so placing the 16 bits in
    the high half of a 32-bit word gives the same number as a float32.
    """
    b = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):      # NaN payloads widen as NaN
        return b.view(np.float32).astype(np.float64)


def f32_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of IEEE binary32 bit patterns (uint32) as float64."""
    return np.asarray(bits).astype(np.uint32).view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits and binary32's exponent range.  For a
    normal value with |x| in [2^e, 2^(e+1)) the spacing of bfloat16 numbers
    is 2^(e-7); below 2^-126 the spacing is the fixed subnormal quantum
    2^-133.  The value is divided by its spacing (exact: a power of two),
    rounded to the nearest integer with ties to even (``np.rint``) and
    scaled back.  Results at or beyond 2^128 overflow to infinity.  NaN and
    infinities pass through.  One rounding step only: no detour via float32.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    finite = np.isfinite(x) & (x != 0.0)
    xf = x[finite]
    _, e = np.frexp(np.abs(xf))           # |x| = m * 2^e, m in [0.5, 1)
    e = e.astype(np.int64) - 1            # |x| in [2^e, 2^(e+1))
    spacing_exp = np.maximum(e - 7, -133)
    q = np.ldexp(1.0, spacing_exp)
    r = np.rint(xf / q) * q
    r[np.abs(r) >= 2.0 ** 128] = np.inf * np.sign(r[np.abs(r) >= 2.0 ** 128])
    out[finite] = r
    return out


def bf16_from_f64_bits(x: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) of float64 values that are already
    bfloat16 numbers (for example the output of :func:`round_to_bf16`).

    Such a value is exactly a float32 whose low 16 bits are zero, so the bit
    pattern is the float32 pattern shifted right by 16.
    """
    x = np.asarray(x, dtype=np.float64)
    nan = np.isnan(x)
    f = np.where(nan, 0.0, x).astype(np.float32)
    u = f.view(np.uint32)
    if not np.array_equal(f.astype(np.float64), np.where(nan, 0.0, x)) or np.any((u & np.uint32(0xFFFF)) != 0):
        raise ValueError("value is not representable in bfloat16")
    bits = (u >> np.uint32(16)).astype(np.uint16)
    bits[nan] = np.uint16(0x7FC0)          # one quiet NaN stands for every NaN
    return bits


# ---------------------------------------------------------------------------
# Shard layouts (page "Nano-vLLM walkthrough 22", §2-§5; page "Tensor
# parallelism from scratch", tp.py).  Weights are stored [out, in], so that a
# linear layer computes x @ W^T: a column split (on the output dimension)
# takes rows, a row split (on the input dimension) takes columns.
# ---------------------------------------------------------------------------

def divide(numerator: int, denominator: int) -> int:
    """Exact integer division; a split that does not divide evenly is an
    error (Nano-vLLM walkthrough 22, §1 ``divide``)."""
    if numerator % denominator != 0:
        raise ValueError(f"{numerator} is not divisible by {denominator}")
    return numerator // denominator


def column_shard(w_full: np.ndarray, t: int, r: int) -> np.ndarray:
    """Rank r's rows of a column-parallel weight [out, in]: rows
    [r*out/t, (r+1)*out/t) (Nano-vLLM walkthrough 22, §3 ColumnParallelLinear:
    shard_size = out/t, start = rank*shard_size, narrow on dim 0).  The same
    cut applies to a 1-D bias of length out."""
    size = divide(w_full.shape[0], t)
    return w_full[r * size:(r + 1) * size]


def row_shard(w_full: np.ndarray, t: int, r: int) -> np.ndarray:
    """Rank r's columns of a row-parallel weight [out, in]: columns
    [r*in/t, (r+1)*in/t) (Nano-vLLM walkthrough 22, §4 RowParallelLinear:
    narrow on dim 1).  A row-parallel bias is not split."""
    size = divide(w_full.shape[1], t)
    return w_full[:, r * size:(r + 1) * size]


def merged_column_shard(parts: Sequence[np.ndarray], t: int, r: int) -> np.ndarray:
    """Rank r's block of a merged column-parallel weight (gate_up or q/k/v).

    Nano-vLLM walkthrough 22, §5 "double cut": the merged table holds the
    parts one after another, each part cut into t chunks along its output
    dimension; rank r keeps chunk r of every part, in part order.  Part p
    therefore sits at row offset sum(sizes[:p])/t of the rank's block and
    spans sizes[p]/t rows.  For gate_up this is [gate rows of rank r ; up
    rows of rank r], NOT a contiguous split of [gate; up].
    """
    blocks = []
    for p in parts:
        size = divide(p.shape[0], t)
        blocks.append(p[r * size:(r + 1) * size])
    return np.concatenate(blocks, axis=0)


def qkv_shard(wq: np.ndarray, wk: np.ndarray, wv: np.ndarray, num_heads: int,
              num_kv_heads: int, head_size: int, t: int, r: int) -> np.ndarray:
    """Rank r's block of a merged QKV weight (Nano-vLLM walkthrough 22, §5
    QKVParallelLinear): per rank, num_heads/t query heads, then
    num_kv_heads/t key heads, then as many value heads, each head being
    head_size consecutive rows.  The head counts must divide by t."""
    nh = divide(num_heads, t)
    nkv = divide(num_kv_heads, t)
    assert wq.shape[0] == num_heads * head_size
    assert wk.shape[0] == num_kv_heads * head_size and wv.shape[0] == wk.shape[0]
    q = wq[r * nh * head_size:(r + 1) * nh * head_size]
    k = wk[r * nkv * head_size:(r + 1) * nkv * head_size]
    v = wv[r * nkv * head_size:(r + 1) * nkv * head_size]
    return np.concatenate([q, k, v], axis=0)


def kv_head_of_rank(num_kv_heads: int, t: int, r: int) -> List[int]:
    """KV heads held by rank r of a head-parallel GQA attention.

    6.2 Tensor-parallel inference, §2.2: with t <= num_kv_heads every rank
    holds num_kv_heads/t distinct KV heads; with t > num_kv_heads every rank
    holds one KV head and each KV head is replicated on t/num_kv_heads ranks
    (t must be divisible by num_kv_heads).  Which rank holds which head is
    in a missing figure; reading taken: consecutive ranks share a head, rank
    r holds head r // (t/num_kv_heads), which is the head its own query
    heads use under GQA grouping (query head q uses KV head
    q // (num_heads/num_kv_heads)).
    """
    if t <= num_kv_heads:
        per = divide(num_kv_heads, t)
        return list(range(r * per, (r + 1) * per))
    return [r // divide(t, num_kv_heads)]


def qkv_shard_gqa(wq: np.ndarray, wk: np.ndarray, wv: np.ndarray, num_heads: int, num_kv_heads: int,
                  head_size: int, t: int, r: int) -> np.ndarray:
    """Rank r's merged [q; k; v] block when the KV heads may be replicated
    (see :func:`kv_head_of_rank`); equals :func:`qkv_shard` when t divides
    the KV head count."""
    nh = divide(num_heads, t)
    q = wq[r * nh * head_size:(r + 1) * nh * head_size]
    heads = kv_head_of_rank(num_kv_heads, t, r)
    k = np.concatenate([wk[h * head_size:(h + 1) * head_size] for h in heads], axis=0)
    v = np.concatenate([wv[h * head_size:(h + 1) * head_size] for h in heads], axis=0)
    return np.concatenate([q, k, v], axis=0)


def vocab_range(vocab: int, t: int, r: int) -> Tuple[int, int]:
    """Token-id range [start, end) owned by rank r of a vocab-parallel table.

    Tensor parallelism from scratch, tp.py VocabParallelEmbedding:
    per = ceil(V/t), start = r*per, end = min((r+1)*per, V).  The other pages
    split V/2 per rank for t=2; all rules agree when t divides V.  A rank
    whose start is at or past V owns an empty range.
    """
    per = (vocab + t - 1) // t
    start = min(r * per, vocab)
    end = min((r + 1) * per, vocab)
    return start, end


# ---------------------------------------------------------------------------
# Linear layers and the MLP.
# ---------------------------------------------------------------------------

def linear(x: np.ndarray, w: np.ndarray, b: np.ndarray | None = None) -> np.ndarray:
    """y = x @ w^T (+ b), with w stored [out, in] (Nano-vLLM walkthrough 22,
    §2: the forward of a linear layer is x @ weight.T)."""
    y = np.asarray(x, np.float64) @ np.asarray(w, np.float64).T
    if b is not None:
        y = y + np.asarray(b, np.float64)
    return y


def silu(x: np.ndarray) -> np.ndarray:
    """silu(x) = x * sigmoid(x) = x / (1 + exp(-x)).  The pages name SiLU as
    the activation of Llama/Qwen MLPs (vLLM source analysis 13, §2.2.1; tp.py
    TPMLP) without a formula; this is the standard definition.  Written with
    the sign split so that exp never overflows."""
    x = np.asarray(x, np.float64)
    out = np.empty_like(x)
    pos = x >= 0
    out[pos] = x[pos] / (1.0 + np.exp(-x[pos]))
    ex = np.exp(x[~pos])
    out[~pos] = x[~pos] * ex / (1.0 + ex)
    return out


def gelu_tanh(x: np.ndarray) -> np.ndarray:
    """GeLU, tanh approximation, as the numpy demo of vLLM source analysis 13,
    §2.2.2 defines it: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    x = np.asarray(x, np.float64)
    return 0.5 * x * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))


def glu(gate: np.ndarray, up: np.ndarray, act: str) -> np.ndarray:
    """The gated activation between the two MLP matmuls: act(gate) * up
    (tp.py TPMLP: silu(gate_proj(x)) * up_proj(x)).  act is "silu" or
    "gelu_tanh" (the latter an option of this library; both activations are
    pinned to torch's own and to closed-form identities)."""
    if act == "silu":
        return silu(gate) * up
    if act == "gelu_tanh":
        return gelu_tanh(gate) * up
    raise ValueError(act)


def mlp_unsharded(x, w_gate, w_up, w_down, bias=None, act="silu") -> np.ndarray:
    """The plain MLP on one device: Y = act(X Wg^T) * (X Wu^T) @ Wd^T (+ b).

    Weights are stored [out, in]: w_gate, w_up [f, h]; w_down [h, f].
    This is the definition the sharded layer must reproduce (6.2
    Tensor-parallel inference, §1: the sum over shards equals the original).
    """
    g = linear(x, w_gate)
    u = linear(x, w_up)
    return linear(glu(g, u, act), w_down, bias)


def mlp_shard_partials(x, w_gate, w_up, w_down, t, bias=None, act="silu") -> List[np.ndarray]:
    """The t row-parallel partial sums of the tensor-parallel MLP.

    6.2 Tensor-parallel inference, §1: rank i computes act(X A_i) B_i, a full
    n x h partial; A (gate/up) is cut on its output dimension and B (down) on
    its input dimension, with the same cut on the intermediate dimension f.
    The merged gate_up block of rank i is [gate_i; up_i] (double cut).  The
    bias of the row-parallel layer is added by rank 0 only (Nano-vLLM
    walkthrough 22, §4: only rank 0 adds it so that the sum counts it once).
    """
    f = w_gate.shape[0]
    fs = divide(f, t)
    partials = []
    for i in range(t):
        gu = merged_column_shard([w_gate, w_up], t, i)      # [2 f/t, h]
        g = linear(x, gu[:fs])
        u = linear(x, gu[fs:])
        h_i = glu(g, u, act)                                # [n, f/t], stays on rank i
        b_i = row_shard(w_down, t, i)                       # [h, f/t]
        partials.append(linear(h_i, b_i, bias if i == 0 else None))
    return partials


def mlp_sharded(x, w_gate, w_up, w_down, t, bias=None, act="silu", order="direct") -> np.ndarray:
    """Sum of the t partials of :func:`mlp_shard_partials`, in fp64, either in
    rank order ("direct", the one-shot all-reduce) or in ring order ("ring",
    each chunk folded starting at its own index; see :func:`ring_allreduce`)."""
    parts = mlp_shard_partials(x, w_gate, w_up, w_down, t, bias, act)
    if order == "direct":
        return reduce_direct(parts)
    if order == "ring":
        bufs, _ = ring_allreduce(parts, hop="f64")
        return bufs[0]
    raise ValueError(order)


def round_to_f32(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest IEEE binary32 value, ties to even
    (numpy's float64 -> float32 conversion), returned as float64."""
    return np.asarray(x, np.float64).astype(np.float32).astype(np.float64)


def mlp_sharded_rounded(x, w_gate, w_up, w_down, t, bias=None, act="silu", partial_dtype="bf16",
                        order="direct") -> Dict[str, object]:
    """The tensor-parallel MLP with the intermediate results stored in the
    number formats a rank keeps them in.

    6.2 Tensor-parallel inference, §1: rank i computes act(X A_i) B_i; the
    ranks exchange their partials as 2-byte values ("Tensor parallelism from
    scratch", the cost of communication: 2 bytes per element on the wire).
    Reading taken where the pages are silent: every product is exact (fp64
    here), the activation output H_i = act(G_i) * U_i is rounded once to
    bfloat16 (the dtype of the next GEMM's input), each partial
    P_i = H_i B_i^T (+ bias on rank 0, before rounding) is rounded once to
    ``partial_dtype`` ("bf16" or "f32"), and the partials are summed:

    * order "direct": in rank order, exactly (fp64);
    * order "ring": the ring all-reduce of :func:`ring_allreduce`, every hop
      rounded to the partial dtype (a ring over a bf16 wire rounds at each
      hop);
    * partial_dtype None ("fused"): no partial exists; Y = sum_i H_i B_i^T
      (+ bias once), exact.

    Returns a dict: ``y`` [n, h]; ``h`` / ``h_exact`` the t rounded and
    unrounded H_i; ``p`` the t rounded partials (empty when fused) and
    ``p_exact`` the t products H_i B_i^T (+ bias on rank 0) before rounding.
    """
    f = w_gate.shape[0]
    fs = divide(f, t)
    hs, hs_exact, ps, ps_exact = [], [], [], []
    for i in range(t):
        gu = merged_column_shard([w_gate, w_up], t, i)
        h_exact = glu(linear(x, gu[:fs]), linear(x, gu[fs:]), act)
        h_i = round_to_bf16(h_exact)
        hs_exact.append(h_exact)
        hs.append(h_i)
        ps_exact.append(linear(h_i, row_shard(w_down, t, i), bias if i == 0 else None))
    if partial_dtype is None:
        return {"y": reduce_direct(ps_exact), "h": hs, "h_exact": hs_exact, "p": [], "p_exact": ps_exact}
    rnd = {"bf16": round_to_bf16, "f32": round_to_f32}[partial_dtype]
    ps = [rnd(p) for p in ps_exact]
    if order == "direct":
        y = reduce_direct(ps)
    elif order == "ring":
        bufs, _ = ring_allreduce(ps, hop=partial_dtype)
        y = bufs[0]
    else:
        raise ValueError(order)
    return {"y": y, "h": hs, "h_exact": hs_exact, "p": ps, "p_exact": ps_exact}


# ---------------------------------------------------------------------------
# The all-reduce (sum) of the partials.
# ---------------------------------------------------------------------------

def reduce_direct(partials: Sequence[np.ndarray]) -> np.ndarray:
    """One-shot all-reduce: out = 0; for each peer buffer, out += buffer
    (vLLM source analysis 13, low-latency all-reduce pseudocode after §1.2).
    Summed in rank order, in float64."""
    out = np.zeros_like(np.asarray(partials[0], np.float64))
    for p in partials:
        out = out + np.asarray(p, np.float64)
    return out


def reduce_direct_f32(partials: Sequence[np.ndarray]) -> np.ndarray:
    """The same rank-order sum carried in IEEE binary32 (round to nearest
    even after every add), starting from the first buffer.  Each partial is
    first converted to float32 (exact for bfloat16 and float32 inputs).
    Returned as float64 holding float32 values."""
    acc = np.asarray(partials[0], np.float64).astype(np.float32)
    for p in partials[1:]:
        acc = (acc + np.asarray(p, np.float64).astype(np.float32)).astype(np.float32)
    return acc.astype(np.float64)


def ring_chunks(count: int, n: int) -> List[Tuple[int, int]]:
    """The N chunks of a K-element buffer in the ring all-reduce: chunk c is
    [c*ceil(K/N), min((c+1)*ceil(K/N), K)) (vLLM source analysis 13, §1.1.1:
    the data is cut into N chunks of about K/N elements).  Chunks past the
    end are empty."""
    cs = (count + n - 1) // n if n > 0 else 0
    return [(min(c * cs, count), min((c + 1) * cs, count)) for c in range(n)]


def ring_schedule(n: int) -> List[Tuple[str, int, int, int, int]]:
    """Who sends which chunk to whom at each step of a ring all-reduce.

    vLLM source analysis 13, §1.1.1 and §1.1.2: the N ranks form a logical
    ring and each talks only to its neighbour.  In each of the N-1
    reduce-scatter steps every rank sends one chunk and receives one,
    adding the received chunk into its own copy; the updated chunk is what
    travels on the next step.  Then N-1 all-gather steps pass the finished
    chunks around the ring, copying instead of adding.

    The figures that fix which chunk a rank sends first are missing from the
    page.  Reading taken: at reduce-scatter step s rank r sends chunk
    (r - s) mod N to rank (r + 1) mod N, so every chunk starts at the rank of
    its own index and rank r ends holding the finished chunk (r + 1) mod N;
    at all-gather step s rank r sends chunk (r + 1 - s) mod N.

    Returns (phase, step, sender, receiver, chunk) tuples.
    """
    steps = []
    for s in range(n - 1):
        for r in range(n):
            steps.append(("reduce_scatter", s, r, (r + 1) % n, (r - s) % n))
    for s in range(n - 1):
        for r in range(n):
            steps.append(("all_gather", s, r, (r + 1) % n, (r + 1 - s) % n))
    return steps


def _hop_add(a: np.ndarray, b: np.ndarray, hop: str) -> np.ndarray:
    """One reduce-scatter addition, rounded to the buffer's number format:
    "f64" (no rounding), "f32" (binary32 add, ties to even) or "bf16"
    (exact sum of two bfloat16 values, then one rounding to bfloat16)."""
    if hop == "f64":
        return a + b
    if hop == "f32":
        return (a.astype(np.float32) + b.astype(np.float32)).astype(np.float32).astype(np.float64)
    if hop == "bf16":
        return round_to_bf16(a + b)
    raise ValueError(hop)


def ring_allreduce(partials: Sequence[np.ndarray], hop: str = "f64") -> Tuple[List[np.ndarray], Dict[str, object]]:
    """Simulate the ring all-reduce of :func:`ring_schedule` by message
    passing between N rank buffers (each a flattened copy of one partial).

    All sends of a step happen at once: every message is read from the
    sender's buffer as it was before the step, then delivered.  hop selects
    how each reduce-scatter addition rounds (see ``_hop_add``); with
    hop="f32" the buffers hold binary32 values throughout.

    Returns the N buffers after the all-gather, reshaped like the input, and
    a dict with the number of communication steps, the number of elements
    each rank sent, the chunk bounds and the buffers as they stood after
    the reduce-scatter phase.
    """
    n = len(partials)
    shape = np.asarray(partials[0]).shape
    bufs = [np.asarray(p, np.float64).reshape(-1).copy() for p in partials]
    if hop == "f32":
        bufs = [b.astype(np.float32).astype(np.float64) for b in bufs]
    count = bufs[0].size
    chunks = ring_chunks(count, n)
    sent = [0] * n
    phases_seen = []
    sched = ring_schedule(n)
    after_rs = None
    for phase in ("reduce_scatter", "all_gather"):
        if phase == "all_gather":
            after_rs = [b.reshape(shape).copy() for b in bufs]
        for s in range(n - 1):
            msgs = []
            for (ph, st, src, dst, c) in sched:
                if ph == phase and st == s:
                    lo, hi = chunks[c]
                    msgs.append((dst, c, bufs[src][lo:hi].copy()))
                    sent[src] += hi - lo
            for dst, c, data in msgs:
                lo, hi = chunks[c]
                if phase == "reduce_scatter":
                    bufs[dst][lo:hi] = _hop_add(bufs[dst][lo:hi], data, hop)
                else:
                    bufs[dst][lo:hi] = data
            phases_seen.append((phase, s))
    stats = {"steps": len(phases_seen), "sent_per_rank": sent, "chunks": chunks,
             "after_reduce_scatter": after_rs}
    return [b.reshape(shape) for b in bufs], stats


def ring_fold_order(n: int, c: int) -> List[int]:
    """The order in which the ring of :func:`ring_schedule` adds the ranks'
    contributions into chunk c: c, c+1, ..., c+N-1 (mod N).  Derived by
    following chunk c through the reduce-scatter steps: rank c sends it at
    step 0, and each receiver adds its own copy and forwards the result."""
    order = [c % n]
    holder = c % n
    for s in range(n - 1):
        nxt = (holder + 1) % n
        order.append(nxt)
        holder = nxt
    return order


# ---------------------------------------------------------------------------
# Vocab-parallel embedding and the sharded LM head.
# ---------------------------------------------------------------------------

def vocab_parallel_embedding(ids: np.ndarray, table: np.ndarray, t: int) -> Tuple[np.ndarray, List[np.ndarray]]:
    """Vocab-parallel input embedding.

    Tensor parallelism from scratch, tp.py VocabParallelEmbedding; vLLM
    source analysis 13, §2.4.1: rank r holds rows [start_r, end_r) of the
    table (:func:`vocab_range`).  It looks up id - start_r for the ids in its
    range, and its output for every other id (including ids below 0 or at or
    past V) is set to exactly 0.0 (masked_fill, not a multiply by the mask,
    so a NaN or Inf row of another rank never leaks in).  The t outputs are
    then summed (the all-reduce), in rank order, starting from rank 0's
    output.

    Returns (sum, per-rank outputs), float64.
    """
    ids = np.asarray(ids, dtype=np.int64)
    table = np.asarray(table, np.float64)
    vocab, h = table.shape
    partials = []
    for r in range(t):
        start, end = vocab_range(vocab, t, r)
        local = table[start:end]
        mask = (ids < start) | (ids >= end)
        safe = np.where(mask, 0, ids - start)
        out = np.zeros(ids.shape + (h,), np.float64)
        if local.shape[0] > 0:
            out = local[safe]
        out = np.where(mask[..., None], 0.0, out)
        partials.append(out)
    total = partials[0].copy()
    for p in partials[1:]:
        total = total + p
    return total, partials


def lm_head_sharded(x: np.ndarray, table: np.ndarray, t: int) -> Tuple[np.ndarray, List[np.ndarray]]:
    """Vocab-sharded LM head.  vLLM source analysis 13, §2.4.2: rank r
    computes Y_r = X E_r^T with E_r its [V/t, h] slice of the (tied) table;
    the Y_r are gathered and concatenated along the vocab dimension (tp.py
    TPTransformer: all_gather, cat on the last dim, slice [:V]).  Returns
    (concatenated logits [n, V], per-rank logits), float64."""
    vocab = table.shape[0]
    parts = []
    for r in range(t):
        start, end = vocab_range(vocab, t, r)
        parts.append(linear(x, table[start:end]))
    return shard_gather(parts)[:, :vocab], parts


def lm_head_unsharded(x: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Single-device logits X E^T, the definition the sharded head must
    reproduce."""
    return linear(x, table)


def shard_gather(parts: Sequence[np.ndarray]) -> np.ndarray:
    """All-gather of vocab-sharded logits: the t [n, cols_r] blocks
    concatenated along the last dimension in rank order."""
    return np.concatenate([np.asarray(p, np.float64) for p in parts], axis=-1)


# ---------------------------------------------------------------------------
# Sequence parallelism: the all-reduce split into reduce-scatter + all-gather
# around the per-token residual add and RMSNorm (page "Tensor parallelism from
# scratch", exercise 1 and its reference answer; the pre-norm residual of
# tp.py TPTransformer: x = x + block(norm(x))).
# ---------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, weight: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last dimension: x / sqrt(mean(x^2) + eps) * weight.

    The pages name RMSNorm (tp.py imports it; "6.2 Tensor-parallel
    inference", §6.2 table: not split, one copy per rank) without giving its
    formula; this is the standard definition.
    """
    x = np.asarray(x, np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(weight, np.float64)


def token_chunks(n: int, t: int) -> List[Tuple[int, int]]:
    """Token rows owned by each rank after the reduce-scatter: rank r gets
    rows [r*ceil(n/t), min((r+1)*ceil(n/t), n)) ("each card gets the full
    result of 1/tp of the tokens")."""
    per = (n + t - 1) // t if t > 0 else 0
    return [(min(r * per, n), min((r + 1) * per, n)) for r in range(t)]


def reduce_scatter_fold_order(n: int, c: int) -> List[int]:
    """Order in which the reduce-scatter ring of :func:`ring_reduce_scatter`
    adds the ranks' copies of chunk c: c+1, c+2, ..., c+N (mod N), so that
    the finished chunk lands on rank c."""
    return [(c + 1 + j) % n for j in range(n)]


def ring_reduce_scatter(partials: Sequence[np.ndarray], chunks: Sequence[Tuple[int, int]] | None = None,
                        hop: str = "f64") -> Tuple[List[np.ndarray], Dict[str, object]]:
    """Reduce-scatter on a ring by message passing (vLLM source analysis 13,
    §1.1.1): N-1 steps; at each step every rank sends one chunk to its right
    neighbour, which adds it into its own copy (rounded as ``_hop_add``).

    Which chunk a rank sends first is not fixed by the page (its figures are
    missing).  For a reduce-scatter whose rank r must end holding chunk r
    (the token rows it owns in sequence parallelism), rank r sends chunk
    (r - s - 1) mod N at step s.  ``chunks`` are (lo, hi) ranges of the
    flattened buffer (default: :func:`ring_chunks`).

    Returns the N buffers after the last step (rank r's chunk r is final; its
    other chunks hold partial sums) and counters.
    """
    n = len(partials)
    shape = np.asarray(partials[0]).shape
    bufs = [np.asarray(p, np.float64).reshape(-1).copy() for p in partials]
    if hop == "f32":
        bufs = [b.astype(np.float32).astype(np.float64) for b in bufs]
    if chunks is None:
        chunks = ring_chunks(bufs[0].size, n)
    sent = [0] * n
    for s in range(n - 1):
        msgs = []
        for r in range(n):
            c = (r - s - 1) % n
            lo, hi = chunks[c]
            msgs.append(((r + 1) % n, c, bufs[r][lo:hi].copy()))
            sent[r] += hi - lo
        for dst, c, data in msgs:
            lo, hi = chunks[c]
            bufs[dst][lo:hi] = _hop_add(bufs[dst][lo:hi], data, hop)
    return [b.reshape(shape) for b in bufs], {"steps": n - 1, "sent_per_rank": sent, "chunks": list(chunks)}


def all_gather_rows(pieces: Sequence[np.ndarray]) -> np.ndarray:
    """All-gather along the token dimension: the ranks' row blocks stacked in
    rank order."""
    return np.concatenate([np.asarray(p, np.float64) for p in pieces], axis=0)


def sequence_parallel_residual_norm(partials: Sequence[np.ndarray], residual: np.ndarray | None,
                                    weight: np.ndarray, eps: float, order: str = "direct"):
    """The sequence-parallel replacement of "all-reduce, then residual add and
    RMSNorm on every token on every rank": reduce-scatter the [n, h]
    partials over token rows, add the residual and apply RMSNorm on each
    rank's own rows only, all-gather the rows.

    order "direct": each rank sums its rows of the t partials in rank order;
    "ring": the reduce-scatter ring above (fp64 adds, so only the order of the
    fold differs).  Returns (new residual [n, h], normed [n, h], per-rank
    (residual, normed) row blocks).
    """
    t = len(partials)
    p64 = [np.asarray(p, np.float64) for p in partials]
    n, h = p64[0].shape
    rows = token_chunks(n, t)
    if order == "ring":
        chunks = [(lo * h, hi * h) for lo, hi in rows]
        bufs, _ = ring_reduce_scatter(p64, chunks=chunks, hop="f64")
        owned = [bufs[r][lo:hi] for r, (lo, hi) in enumerate(rows)]
    elif order == "direct":
        owned = [reduce_direct([p[lo:hi] for p in p64]) for lo, hi in rows]
    else:
        raise ValueError(order)
    res_blocks, norm_blocks = [], []
    for r, (lo, hi) in enumerate(rows):
        x = owned[r] if residual is None else np.asarray(residual, np.float64)[lo:hi] + owned[r]
        res_blocks.append(x)
        norm_blocks.append(rmsnorm(x, weight, eps))
    return all_gather_rows(res_blocks), all_gather_rows(norm_blocks), list(zip(res_blocks, norm_blocks))


# ---------------------------------------------------------------------------
# Cost model used only to annotate results.
# ---------------------------------------------------------------------------

def allreduce_time(size_bytes: float, t: int, bw_bytes_per_s: float, alpha_s: float = 0.0) -> float:
    """T = alpha + 2 (t-1)/t * S / B  (6.2 Tensor-parallel inference, §3.1)."""
    return alpha_s + 2.0 * (t - 1) / t * size_bytes / bw_bytes_per_s
