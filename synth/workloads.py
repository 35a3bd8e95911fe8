"""Seeded synthetic workloads shaped like the pages' few-shot, branching, multi-turn and fork
programs. Each builder returns token sequences and their structure only; no cache or attention
arithmetic happens here.

Token ids are uniform in [0, 32000). Where a builder needs two sibling branches to diverge at a
given position, it redraws the first token of the later branch until it differs (the redraw
stream is part of the builder's definition). No public benchmark item is used: the shapes stand
in for MMLU 5-shot, HellaSwag, multi-turn chat, tree-of-thought and self-consistency programs.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import irwin_hall_normal, permutation, tokens, uniform_int


@dataclass
class Model:
    layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    dtype: str          # "bf16" or "f32"
    seed: int = 0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def sm_scale(self) -> float:
        return 1.0 / float(np.sqrt(self.head_dim))


@dataclass
class Phase:
    """kind: 'extend' (compute the unmatched suffix of each sequence), 'cache' (insert sequences
    one at a time as already computed; their KV is written straight into the pool), 'decode'
    (one new token per
    request over its cached context: seqs are full sequences, context = all but the last token)."""
    kind: str
    seqs: list
    keep_locked: bool = False


@dataclass
class Workload:
    name: str
    model: Model
    pool_slots: int
    pool_order: np.ndarray | None       # initial free-list order (None = identity)
    phases: list = field(default_factory=list)
    max_ctx: int = 0                    # slot-table row length (multiple of 16)
    notes: dict = field(default_factory=dict)


def _first_distinct(seed, seq, taken, redraw_stream):
    """Redraw seq[0] from `redraw_stream` until it is not in `taken`; returns seq."""
    seq = np.array(seq, dtype=np.int32)
    attempt = 0
    while int(seq[0]) in taken:
        seq[0] = tokens(seed, redraw_stream, 1, start=attempt)[0]
        attempt += 1
    taken.add(int(seq[0]))
    return seq


def _round16(n):
    return (int(n) + 15) // 16 * 16


def tiny_extend(seed: int = 0) -> Workload:
    """1 layer, 2 heads (MHA) x 64, fp32, pool 4096 slots in identity order. Four requests share a
    64-token prefix and have 16 unique suffix tokens each; the first request prefills all 80
    tokens alone, the other three then reuse the 64 cached prefix slots."""
    m = Model(1, 2, 2, 64, "f32", seed)
    prefix = tokens(seed, 1, 64)
    taken = set()
    sufs = [_first_distinct(seed, tokens(seed, 100 + k, 16), taken, 200 + k) for k in range(4)]
    seqs = [np.concatenate([prefix, s]) for s in sufs]
    w = Workload("tiny_extend", m, 4096, None, max_ctx=_round16(80))
    w.phases = [Phase("extend", seqs[:1]), Phase("extend", seqs[1:])]
    return w


def few_shot_extend(seed: int = 0, n_requests: int = 64, prefix_len: int = 2000,
                    suffix_len: int = 50, pool_slots: int = 200_000) -> Workload:
    """Llama-2-7B attention shape (32 x 128 MHA, bf16), 1 layer. A warm request prefills the
    shared few-shot prefix and inserts it; then `n_requests` requests (prefix + unique suffix)
    match the prefix and extend their suffix. Pool free list in seeded random order."""
    m = Model(1, 32, 32, 128, "bf16", seed)
    prefix = tokens(seed, 1, prefix_len)
    taken = set()
    sufs = [_first_distinct(seed, tokens(seed, 100 + k, suffix_len), taken, 10_000 + k)
            for k in range(n_requests)]
    seqs = [np.concatenate([prefix, s]) for s in sufs]
    w = Workload("few_shot_extend", m, pool_slots, permutation(seed, pool_slots),
                 max_ctx=_round16(prefix_len + suffix_len))
    w.phases = [Phase("extend", [prefix]), Phase("extend", seqs)]
    return w


def two_level_extend(seed: int = 0, n_stems: int = 16, n_cont: int = 4, prefix_len: int = 1000,
                     stem_len: int = 100, cont_len: int = 20, distract_len: int = 20,
                     pool_slots: int = 500_000) -> Workload:
    """Llama-2-70B GQA attention (64 q / 8 kv heads x 128, bf16), 1 layer. Leaves are
    prefix + stem_s + cont_{s,c}. Warm-up: the prefix alone, then per stem the prefix, the first
    v_s stem tokens (v_s uniform in 1..99) and distractor tokens, so that each leaf's match ends
    inside a cached edge at a random position (the node splits there). Then all leaves extend."""
    m = Model(1, 64, 8, 128, "bf16", seed)
    prefix = tokens(seed, 1, prefix_len)
    taken = set()
    stems = [_first_distinct(seed, tokens(seed, 100 + s, stem_len), taken, 20_000 + s)
             for s in range(n_stems)]
    v = uniform_int(seed, 300, n_stems, 1, stem_len - 1)
    warm = []
    for s in range(n_stems):
        d = _first_distinct(seed, tokens(seed, 400 + s, distract_len),
                            {int(stems[s][v[s]])}, 30_000 + s)
        warm.append(np.concatenate([prefix, stems[s][: v[s]], d]))
    leaves = []
    for s in range(n_stems):
        taken_c = set()
        for c in range(n_cont):
            cont = _first_distinct(seed, tokens(seed, 1000 + n_cont * s + c, cont_len), taken_c,
                                   40_000 + n_cont * s + c)
            leaves.append(np.concatenate([prefix, stems[s], cont]))
    w = Workload("two_level_extend", m, pool_slots, permutation(seed, pool_slots),
                 max_ctx=_round16(prefix_len + stem_len + cont_len + distract_len))
    w.phases = [Phase("extend", [prefix]), Phase("extend", warm), Phase("extend", leaves)]
    w.notes["v"] = v.tolist()
    return w


def decode_lengths_lognormal(seed: int, n: int, median: int = 2048, lo: int = 128,
                             hi: int = 16384) -> np.ndarray:
    """clip(round(median * exp(z)), lo, hi), z ~ N(0, 1) (Irwin-Hall(4) approximation)."""
    z = irwin_hall_normal(seed, 10, n)
    return np.clip(np.rint(median * np.exp(z)), lo, hi).astype(np.int64)


def multi_turn_decode(seed: int = 0, n_requests: int = 256, branching: int = 4, depth: int = 3,
                      shared: bool = True, lengths=None) -> Workload:
    """Mixtral-8x7B attention (32 q / 8 kv heads x 128, bf16), 1 layer. `n_requests` requests with
    lognormal context lengths (median 2048, clipped to 128..16384) share tree-structured prefixes:
    `branching`**depth internal nodes, each deepest node with `branching` request leaves; a
    depth-k node's segment is floor(min length in its subtree / 4) tokens, the rest of a request
    is its own. Each request decodes one new token (its last token) over its cached context.
    shared=False gives the unshared twin: the same lengths, all tokens unique."""
    m = Model(1, 32, 8, 128, "bf16", seed)
    L = decode_lengths_lognormal(seed, n_requests) if lengths is None else np.asarray(lengths)
    seqs = []
    if shared:
        per_leaf = n_requests // (branching ** depth)
        assert per_leaf * branching ** depth == n_requests
        # node path of request r: digits (r // per_leaf) in base `branching`, most significant first
        segs = {}
        taken_at = {}
        for r in range(n_requests):
            parts = []
            leaf_group = r // per_leaf
            for k in range(1, depth + 1):
                path = tuple((leaf_group // branching ** (depth - i)) % branching
                             for i in range(1, k + 1))
                if path not in segs:
                    # members of this node's subtree
                    span = branching ** (depth - k) * per_leaf
                    first = (leaf_group // branching ** (depth - k)) * span
                    seg_len = int(L[first:first + span].min()) // 4
                    node_id = sum((p + 1) * (branching + 1) ** i for i, p in enumerate(path))
                    tk = taken_at.setdefault(path[:-1], set())
                    segs[path] = _first_distinct(seed, tokens(seed, 2000 + node_id, seg_len),
                                                 tk, 50_000 + node_id)
                parts.append(segs[path])
            used = sum(len(p) for p in parts)
            tk = taken_at.setdefault(("leaf", leaf_group), set())
            own = _first_distinct(seed, tokens(seed, 5000 + r, int(L[r]) - used), tk, 60_000 + r)
            seqs.append(np.concatenate(parts + [own]).astype(np.int32))
    else:
        for r in range(n_requests):
            seqs.append(tokens(seed, 9000 + r, int(L[r])))
    distinct = _distinct_prefix_tokens([s[:-1] for s in seqs])
    pool = int(distinct * 1.1) + n_requests
    w = Workload("multi_turn_decode" + ("" if shared else "_unshared"), m, pool,
                 permutation(seed, pool), max_ctx=_round16(int(L.max())))
    w.phases = [Phase("cache", [s[:-1] for s in seqs]), Phase("decode", seqs)]
    w.notes["lengths"] = L.tolist()
    w.notes["distinct_context_tokens"] = distinct
    return w


def _distinct_prefix_tokens(seqs) -> int:
    """Number of distinct (prefix-identified) token positions: size of the per-token trie."""
    seen = set()
    for s in seqs:
        h = 0
        for t in s.tolist():
            h = hash((h, t))
            seen.add(h)
    return len(seen)


@dataclass
class ForkMixed:
    """The fork / self-consistency mixed step: setup phases, then per-step batches."""
    workload: Workload
    programs: list           # 16 program prefixes (1500 tokens each)
    decode_seqs: list        # 128 decode requests: full sequence at step 0 (last = new token)
    n_forks: int
    suffix_len: int
    seed: int

    def extend_seqs(self, step: int) -> list:
        """prefix_p + a fresh 200-token fork suffix for each program p and fork f at `step`."""
        out = []
        for p, pre in enumerate(self.programs):
            taken = set()
            for f in range(self.n_forks):
                sid = 1_000_000 + step * 1000 + self.n_forks * p + f
                suf = _first_distinct(self.seed, tokens(self.seed, sid, self.suffix_len), taken,
                                      sid + 500_000)
                out.append(np.concatenate([pre, suf]).astype(np.int32))
        return out

    def decode_step_seqs(self, step: int) -> list:
        """Decode request r at `step`: its step-0 sequence plus `step` generated tokens."""
        if step == 0:
            return self.decode_seqs
        return [np.concatenate([s, tokens(self.seed, 70_000 + r, step)]).astype(np.int32)
                for r, s in enumerate(self.decode_seqs)]


def fork_mixed_step(seed: int = 0, layers: int = 32, pool_slots: int = 300_000,
                    n_programs: int = 16, prefix_len: int = 1500, n_forks: int = 5,
                    suffix_len: int = 200, n_decode: int = 128, dec_lo: int = 512,
                    dec_hi: int = 8192, free_at_start: int = 4096, max_steps: int = 64,
                    filler_len: int = 1000) -> ForkMixed:
    """32 layers of Llama-2-7B attention (32 x 128 MHA, bf16), pool 300k slots per layer.
    Decode: 128 requests, lengths uniform in 512..8192; sorted, consecutive fours form fork
    groups sharing their shortest member's context. Extend: 16 programs whose 1500-token prefix
    was cached beforehand (the fork hint), each forking 5 ways with 200 new tokens per step.
    The pool is filled with unreferenced cached leaves (older than everything else) so that only
    `free_at_start` slots are free when the first step starts: eviction runs every step."""
    m = Model(layers, 32, 32, 128, "bf16", seed)
    L = np.sort(uniform_int(seed, 20, n_decode, dec_lo, dec_hi))
    dec = []
    for g in range(n_decode // 4):
        grp = L[4 * g: 4 * g + 4]
        shared = tokens(seed, 3000 + g, int(grp[0]) - 1)
        taken = set()
        for i, Lr in enumerate(grp):
            r = 4 * g + i
            own = tokens(seed, 6000 + r, int(Lr) - len(shared))
            if len(own) > 1:
                own = _first_distinct(seed, own, taken, 80_000 + r)
            dec.append(np.concatenate([shared, own]).astype(np.int32))
    taken = set()
    programs = [_first_distinct(seed, tokens(seed, 100 + p, prefix_len), taken, 90_000 + p)
                for p in range(n_programs)]
    contexts = [s[:-1] for s in dec]
    used = _distinct_prefix_tokens(contexts) + n_programs * prefix_len
    n_fill = pool_slots - free_at_start - used
    assert n_fill >= 0, "decode contexts and programs do not fit the pool"
    filler = []
    i = 0
    while n_fill > 0:
        ln = min(filler_len, n_fill)
        filler.append(_first_distinct(seed, tokens(seed, 200_000 + i, ln), taken, 300_000 + i))
        n_fill -= ln
        i += 1
    w = Workload("fork_mixed_step", m, pool_slots, permutation(seed, pool_slots),
                 max_ctx=_round16(max(int(L.max()) + max_steps, prefix_len + suffix_len)))
    w.phases = [Phase("cache", filler), Phase("cache", programs),
                Phase("cache", contexts, keep_locked=True)]
    w.notes.update(lengths=L.tolist(), filler_tokens=sum(len(f) for f in filler),
                   distinct_decode_context=used - n_programs * prefix_len)
    return ForkMixed(w, programs, dec, n_forks, suffix_len, seed)


def tree_extend(seed: int = 0, root_len: int = 1024, n_branches: int = 16,
                branch_len: int = 1024, per_branch: int = 4, new_len: int = 16,
                pool_slots: int = 100_000) -> Workload:
    """A two-level sharing tree (32 x 128 MHA bf16, 1 layer): a `root_len`-token system prompt
    shared by every request, `n_branches` branches that add `branch_len` tokens of their own
    (a document or conversation per branch), `per_branch` requests per branch adding
    `new_len` new tokens each. The root and the branches are cached beforehand; the extend
    batch lists the requests branch by branch."""
    m = Model(1, 32, 32, 128, "bf16", seed)
    root = tokens(seed, 8000, root_len)
    taken = set()
    cache, seqs = [root], []
    for b in range(n_branches):
        br = _first_distinct(seed, tokens(seed, 8100 + b, branch_len), taken, 8300 + b)
        cache.append(np.concatenate([root, br]))
        qt = set()
        for k in range(per_branch):
            own = _first_distinct(seed, tokens(seed, 8500 + per_branch * b + k, new_len), qt,
                                  9500 + per_branch * b + k)
            seqs.append(np.concatenate([root, br, own]))
    w = Workload("tree_extend", m, pool_slots, permutation(seed, pool_slots),
                 max_ctx=_round16(root_len + branch_len + new_len))
    w.phases = [Phase("cache", cache), Phase("extend", seqs)]
    return w


@dataclass
class ProgramQueue:
    """A waiting queue of extend requests (full sequences, queue order) for batch formation."""
    workload: Workload
    seqs: list
    program: np.ndarray          # program index of each request
    max_batch: int
    max_new_tokens: int


def program_queue(seed: int = 0, n_programs: int = 24, prefix_len: int = 2000,
                  n_questions: int = 8, question_len: int = 50, pool_slots: int = 20_000,
                  max_batch: int = 32, max_new_tokens: int = 16_384, layers: int = 1,
                  shared: bool = True) -> ProgramQueue:
    """Few-shot programs (32 x 128 MHA bf16, 1 layer): each of `n_programs` programs has its own
    `prefix_len`-token prefix and `n_questions` questions of `question_len` tokens. Requests
    arrive interleaved, question-major (program 0..n-1 asking question 0, then question 1, ...),
    into a pool that holds fewer prefixes than there are programs. Per batch at most `max_batch`
    requests and `max_new_tokens` computed tokens. `shared=False` is the no-reuse twin: the same
    lengths and order, but every request has a prefix of its own."""
    m = Model(layers, 32, 32, 128, "bf16", seed)
    taken = set()
    prefixes = [_first_distinct(seed, tokens(seed, 5000 + p, prefix_len), taken, 6000 + p)
                for p in range(n_programs)]
    questions = []
    for p in range(n_programs):
        qt = set()
        questions.append([_first_distinct(seed, tokens(seed, 7000 + p * n_questions + q,
                                                       question_len),
                                          qt, 50_000 + p * n_questions + q)
                          for q in range(n_questions)])
    seqs, prog = [], []
    for q in range(n_questions):
        for p in range(n_programs):
            pre = prefixes[p]
            if not shared:
                pre = _first_distinct(seed, tokens(seed, 90_000 + len(seqs), prefix_len), taken,
                                      190_000 + len(seqs))
            seqs.append(np.concatenate([pre, questions[p][q]]))
            prog.append(p)
    w = Workload("program_queue", m, pool_slots, permutation(seed, pool_slots),
                 max_ctx=_round16(prefix_len + question_len))
    return ProgramQueue(w, seqs, np.array(prog, np.int32), max_batch, max_new_tokens)


CONFIGS = {
    "tiny_extend": tiny_extend,
    "few_shot_extend": few_shot_extend,
    "two_level_extend": two_level_extend,
    "multi_turn_decode": multi_turn_decode,
    "fork_mixed_step": fork_mixed_step,
    "tree_extend": tree_extend,
}
