"""Seeded synthetic workloads (test and bench infrastructure).

The pages evaluate on datasets and checkpoints that are not available here
(an 11,668-prompt task set and a WildChat language set for ELDR; WikiText-2,
MATH and Pile-GitHub for GRACE-MoE).  These workloads stand in for them with
the model shapes of the GRACE-MoE model table (OLMoE E=64 k=8 L=16,
DeepSeek-V2-Lite E=64 k=6 L=26, Qwen3-30B-A3B E=128 k=8 L=48) and the
serving parameters of the ELDR page (KV-block signature granularity, D
decoders, tau = 0.1 band, live loads).

Nothing in this module computes any part of the routing method: it only
draws request structure (lengths, domains, prefix donors, KV-block tables,
cache slots), inputs (centroids, loads, idf weights, group maps) and the
keys from which the counter-based generator (``ih12.h``) derives logits.

Host metadata uses ``numpy.random.RandomState`` (a frozen stream) so the
same seed gives the same workload on every machine.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

SEED_BASE = 0x4D4F4552
KEY_POS_BITS = 12  # prompt positions < 4096


@dataclasses.dataclass
class Batch:
    """One batch of requests [r0, r1) of a workload, as the C ABI takes it.

    Token-level arrays cover *computed* tokens only (cached prefix tokens are
    not run through the model in this prefill).
    """
    r0: int
    r1: int
    req_off: np.ndarray        # int32 [R+1], CSR over computed tokens
    tok_key: np.ndarray        # int64 [T], generator content key per token
    tok_dom: np.ndarray        # int32 [T], bias domain per token (-1: none)
    blk_tab: np.ndarray        # int32 [nblk][2] = (tok0, len), KV blocks of computed tokens
    req_blk_off: np.ndarray    # int32 [R+1], CSR of blocks per request
    cache_idx: np.ndarray      # int32 [ncached], cache slots of cached prefix blocks
    req_cache_off: np.ndarray  # int32 [R+1], CSR of cached blocks per request
    insert_slot: np.ndarray    # int32 [nblk], slot for each full computed block, -1 otherwise

    @property
    def R(self) -> int:
        return self.r1 - self.r0

    @property
    def T(self) -> int:
        return int(self.req_off[-1])

    @property
    def nblk(self) -> int:
        return int(self.blk_tab.shape[0])


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    E: int
    k: int
    L: int
    B: int
    R: int
    prompt_len: np.ndarray      # int64 [R]
    cached_blocks: np.ndarray   # int64 [R]
    donor: np.ndarray           # int64 [R], -1 if none
    dom: np.ndarray             # int32 [R], -1 if none
    ndom: int
    bias: float
    bias_mask: np.ndarray       # uint8 [max(ndom,1)][L][E]
    mask: np.ndarray            # int32 [m], sorted distinct layer ids
    D: int
    tau: float
    centroids: np.ndarray       # float32 [D][m*E]
    loads0: np.ndarray          # int32 [D]
    live: bool
    G: int
    group_of: np.ndarray        # int32 [L][E]
    idf: np.ndarray             # float32 [m][E]
    slot_of_block: list         # per request: int64 array of slot ids of its prompt blocks (-1 partial)
    nslots: int
    hidden_dim: int = 0         # gate-GEMM workloads: H
    wgate_scale: float = 0.02
    key_owner_base: int = 0     # token keys of request r are owned by key_owner_base + r

    @property
    def m(self) -> int:
        return int(self.mask.shape[0])

    # ------------------------------------------------------------------ keys
    def prompt_keys(self, r: int) -> np.ndarray:
        """Generator keys of every prompt position of request r (cached prefix included)."""
        n = int(self.prompt_len[r])
        keys = np.empty(n, dtype=np.int64)
        pos = np.arange(n, dtype=np.int64)
        owner = np.full(n, r, dtype=np.int64)
        cur = r
        cut = int(self.cached_blocks[r]) * self.B
        # positions below `cut` belong to the donor chain
        while cut > 0:
            d = int(self.donor[cur])
            owner[:cut] = d
            cur = d
            cut = min(cut, int(self.cached_blocks[cur]) * self.B)
        keys[:] = ((owner + self.key_owner_base) << KEY_POS_BITS) | pos
        return keys

    def computed_tokens(self, r: int) -> int:
        return int(self.prompt_len[r]) - int(self.cached_blocks[r]) * self.B

    # ---------------------------------------------------------------- batches
    def batch(self, r0: int = 0, r1: Optional[int] = None) -> Batch:
        if r1 is None:
            r1 = self.R
        B = self.B
        R = r1 - r0
        comp = np.array([self.computed_tokens(r) for r in range(r0, r1)], dtype=np.int64)
        req_off = np.zeros(R + 1, dtype=np.int64)
        np.cumsum(comp, out=req_off[1:])
        T = int(req_off[-1])
        tok_key = np.empty(T, dtype=np.int64)
        tok_dom = np.empty(T, dtype=np.int32)
        nb = (comp + B - 1) // B
        req_blk_off = np.zeros(R + 1, dtype=np.int64)
        np.cumsum(nb, out=req_blk_off[1:])
        nblk = int(req_blk_off[-1])
        blk_tab = np.empty((nblk, 2), dtype=np.int32)
        insert_slot = np.empty(nblk, dtype=np.int32)
        ncached = self.cached_blocks[r0:r1]
        req_cache_off = np.zeros(R + 1, dtype=np.int64)
        np.cumsum(ncached, out=req_cache_off[1:])
        cache_idx = np.empty(int(req_cache_off[-1]), dtype=np.int32)
        for i, r in enumerate(range(r0, r1)):
            c0 = int(self.cached_blocks[r]) * B
            keys = self.prompt_keys(r)[c0:]
            a, b = int(req_off[i]), int(req_off[i + 1])
            tok_key[a:b] = keys
            tok_dom[a:b] = self.dom[r]
            n = b - a
            j = np.arange(int(nb[i]), dtype=np.int64)
            bb = int(req_blk_off[i])
            blk_tab[bb:bb + len(j), 0] = a + j * B
            blk_tab[bb:bb + len(j), 1] = np.minimum(B, n - j * B)
            slots = self.slot_of_block[r]
            cb = int(self.cached_blocks[r])
            insert_slot[bb:bb + len(j)] = slots[cb:cb + len(j)]
            cache_idx[int(req_cache_off[i]):int(req_cache_off[i + 1])] = slots[:cb]
        return Batch(r0, r1, req_off.astype(np.int32), tok_key, tok_dom, blk_tab,
                     req_blk_off.astype(np.int32), cache_idx,
                     req_cache_off.astype(np.int32), insert_slot)

    def chunks(self, max_tokens: int) -> list:
        """Split the requests into consecutive batches of at most max_tokens computed tokens."""
        out, r0, acc = [], 0, 0
        for r in range(self.R):
            c = self.computed_tokens(r)
            if acc + c > max_tokens and r > r0:
                out.append((r0, r))
                r0, acc = r, 0
            acc += c
        out.append((r0, self.R))
        return out


# ---------------------------------------------------------------------------
# workload recipes
# ---------------------------------------------------------------------------

def _lognormal_lengths(rs, R, median, sigma, lo, hi):
    x = rs.lognormal(mean=np.log(median), sigma=sigma, size=R)
    return np.clip(np.rint(x), lo, hi).astype(np.int64)


def _bias_mask(rs, ndom, L, E, nbias):
    bm = np.zeros((max(ndom, 1), L, E), dtype=np.uint8)
    for d in range(ndom):
        for l in range(L):
            bm[d, l, rs.choice(E, size=nbias, replace=False)] = 1
    return bm


def _centroids(rs, D, ndom, bias_mask, mask, E, noise):
    m = len(mask)
    C = np.empty((D, m * E), dtype=np.float64)
    for d in range(D):
        if ndom > 0:
            g = d % ndom
            base = 1.0 + 2.0 * bias_mask[g][mask].astype(np.float64).reshape(-1)
        else:
            base = np.ones(m * E, dtype=np.float64)
        base /= np.sqrt(np.dot(base, base))
        C[d] = base + rs.normal(0.0, noise, size=m * E)
    return C.astype(np.float32)


def _slots(prompt_len, cached_blocks, donor, B):
    R = len(prompt_len)
    slot_of_block = []
    nxt = 0
    for r in range(R):
        nbp = int((prompt_len[r] + B - 1) // B)
        s = np.full(nbp, -1, dtype=np.int64)
        cb = int(cached_blocks[r])
        if cb:
            s[:cb] = slot_of_block[int(donor[r])][:cb]
        for j in range(cb, nbp):
            if (j + 1) * B <= prompt_len[r]:
                s[j] = nxt
                nxt += 1
        slot_of_block.append(s)
    return slot_of_block, nxt


CONFIGS = ("c1", "c2", "c3", "c4", "c5")


def make_workload(name: str, R: Optional[int] = None, seed: Optional[int] = None) -> Workload:
    """Build workload `name` (c1..c5); `R` overrides the request count (reduced parity cases)."""
    idx = CONFIGS.index(name) + 1
    if seed is None:
        seed = SEED_BASE + idx
    rs = np.random.RandomState(seed & 0xFFFFFFFF)
    B, tau, bias, G = 16, 0.1, 1.5, 8
    prefix_frac = 0.0
    live = False
    H = 0
    if name == "c1":      # OLMoE-shaped tiny
        E, k, L, Rd, ndom, D = 64, 8, 16, 32, 4, 4
        mask = np.arange(L, dtype=np.int32)
    elif name == "c2":    # DeepSeek-V2-Lite-shaped calibration
        E, k, L, Rd, ndom, D = 64, 6, 26, 1000, 4, 16
        mask = np.arange(L, dtype=np.int32)
    elif name == "c3":    # Qwen3-30B-A3B-shaped
        E, k, L, Rd, ndom, D = 128, 8, 48, 1000, 4, 16
        mask = None
    elif name == "c4":    # online routing stream with prefix reuse and live loads
        E, k, L, Rd, ndom, D = 128, 8, 48, 14000, 8, 16
        mask = None
        prefix_frac, live = 0.30, True
    else:                 # c5: gate GEMM feeding the c3-style path
        E, k, L, Rd, ndom, D = 128, 8, 48, 256, 0, 16
        mask = None
        H = 2048
    R = Rd if R is None else int(R)
    if mask is None:
        mask = np.sort(rs.choice(L, size=12, replace=False)).astype(np.int32)

    if name == "c1":
        plen = rs.randint(16, 129, size=R).astype(np.int64)
    elif name == "c2":
        plen = _lognormal_lengths(rs, R, 512, 0.75, 32, 4096)
    elif name == "c3":
        plen = _lognormal_lengths(rs, R, 1024, 0.75, 32, 4096)
    elif name == "c4":
        plen = rs.randint(64, 2049, size=R).astype(np.int64)
    else:
        plen = np.full(R, 2048, dtype=np.int64)

    if name == "c4":
        probs = np.array([0.50, 0.25, 0.10, 0.05, 0.04, 0.03, 0.02, 0.01])
        dom = rs.choice(ndom, size=R, p=probs).astype(np.int32)
    elif ndom > 0:
        dom = rs.randint(0, ndom, size=R).astype(np.int32)
    else:
        dom = np.full(R, -1, dtype=np.int32)

    bias_mask = _bias_mask(rs, ndom, L, E, 3 * E // 16)

    donor = np.full(R, -1, dtype=np.int64)
    cached = np.zeros(R, dtype=np.int64)
    if prefix_frac > 0:
        last_of_group = {}
        seen = {g: [] for g in range(ndom)}
        for r in range(R):
            g = int(dom[r])
            if seen[g] and rs.random_sample() < prefix_frac:
                d = seen[g][rs.randint(0, len(seen[g]))]
                want = rs.randint(4, 65)
                nb = min(want, int(plen[r]) // B - 1, int(plen[d]) // B)
                if nb >= 1:
                    donor[r], cached[r] = d, nb
            seen[g].append(r)
            last_of_group[g] = r

    slot_of_block, nslots = _slots(plen, cached, donor, B)
    centroids = _centroids(rs, D, ndom, bias_mask, mask, E, 0.05)
    loads0 = (np.zeros(D, dtype=np.int32) if live
              else rs.randint(0, 64, size=D).astype(np.int32))
    group_of = np.tile((np.arange(E) * G // E).astype(np.int32), (L, 1))
    idf = (1.0 + 0.5 * rs.random_sample((len(mask), E))).astype(np.float32)
    return Workload(name=name, seed=seed, E=E, k=k, L=L, B=B, R=R, prompt_len=plen,
                    cached_blocks=cached, donor=donor, dom=dom, ndom=ndom, bias=bias,
                    bias_mask=bias_mask, mask=mask, D=D, tau=tau, centroids=centroids,
                    loads0=loads0, live=live, G=G, group_of=group_of, idf=idf,
                    slot_of_block=slot_of_block, nslots=nslots, hidden_dim=H)


CALIB_OWNER_BASE = 1 << 24  # calibration prompts never share a token key with served requests


def make_calibration(wl: Workload, R: int = 1000, seed: Optional[int] = None) -> Workload:
    """The offline calibration prompts of the model that `wl` serves: the same logit
    stream (seed), expert biases per domain and shapes, with R new prompts -- lengths
    lognormal(ln 512, 0.75) clipped to [32, 4096] as in the calibration config, domains
    uniform, no prefix reuse -- whose token keys are distinct from every served request's.
    Every layer is in the mask (the calibration chooses the serving mask)."""
    rs = np.random.RandomState((wl.seed if seed is None else seed) ^ 0xCA11B)
    plen = _lognormal_lengths(rs, R, 512, 0.75, 32, 4096)
    dom = (rs.randint(0, wl.ndom, size=R).astype(np.int32) if wl.ndom > 0
           else np.full(R, -1, dtype=np.int32))
    cached = np.zeros(R, dtype=np.int64)
    donor = np.full(R, -1, dtype=np.int64)
    slot_of_block, nslots = _slots(plen, cached, donor, wl.B)
    mask = np.arange(wl.L, dtype=np.int32)
    return Workload(name=wl.name + "-calibration", seed=wl.seed, E=wl.E, k=wl.k, L=wl.L, B=wl.B, R=R,
                    prompt_len=plen, cached_blocks=cached, donor=donor, dom=dom, ndom=wl.ndom,
                    bias=wl.bias, bias_mask=wl.bias_mask, mask=mask, D=wl.D, tau=wl.tau,
                    centroids=np.zeros((wl.D, wl.L * wl.E), dtype=np.float32), loads0=wl.loads0,
                    live=False, G=wl.G, group_of=wl.group_of,
                    idf=np.ones((wl.L, wl.E), dtype=np.float32), slot_of_block=slot_of_block,
                    nslots=nslots, hidden_dim=wl.hidden_dim, key_owner_base=CALIB_OWNER_BASE)


def make_custom(E: int, k: int, L: int, lengths, *, B: int = 16, mask=None, ndom: int = 2,
                nbias: Optional[int] = None, bias: float = 1.5, D: int = 4, tau: float = 0.1,
                G: int = 4, prefix_frac: float = 0.0, live: bool = False,
                seed: int = 1234) -> Workload:
    """A small workload with explicit shapes (parity edge cases and oracle pins).

    `lengths` are prompt lengths; with `prefix_frac` > 0 a request reuses the
    prefix of an earlier request of the same domain (whole KV blocks, at least
    one computed token left).
    """
    rs = np.random.RandomState(seed & 0xFFFFFFFF)
    plen = np.asarray(lengths, dtype=np.int64)
    R = len(plen)
    mask = np.arange(L, dtype=np.int32) if mask is None else np.asarray(mask, dtype=np.int32)
    dom = rs.randint(0, max(ndom, 1), size=R).astype(np.int32) if ndom > 0 else \
        np.full(R, -1, dtype=np.int32)
    bias_mask = _bias_mask(rs, ndom, L, E, nbias if nbias is not None else max(1, 3 * E // 16))
    donor = np.full(R, -1, dtype=np.int64)
    cached = np.zeros(R, dtype=np.int64)
    if prefix_frac > 0:
        for r in range(1, R):
            cands = [d for d in range(r) if dom[d] == dom[r]]
            if cands and rs.random_sample() < prefix_frac:
                d = cands[rs.randint(0, len(cands))]
                nb = min(rs.randint(1, 5), (int(plen[r]) - 1) // B, int(plen[d]) // B)
                if nb >= 1:
                    donor[r], cached[r] = d, nb
    slot_of_block, nslots = _slots(plen, cached, donor, B)
    centroids = _centroids(rs, D, ndom, bias_mask, mask, E, 0.05)
    loads0 = np.zeros(D, dtype=np.int32) if live else rs.randint(0, 64, size=D).astype(np.int32)
    group_of = np.tile((np.arange(E) * G // E).astype(np.int32), (L, 1))
    idf = (1.0 + 0.5 * rs.random_sample((len(mask), E))).astype(np.float32)
    return Workload(name="custom", seed=seed, E=E, k=k, L=L, B=B, R=R, prompt_len=plen,
                    cached_blocks=cached, donor=donor, dom=dom, ndom=ndom, bias=bias,
                    bias_mask=bias_mask, mask=mask, D=D, tau=tau, centroids=centroids,
                    loads0=loads0, live=live, G=G, group_of=group_of, idf=idf,
                    slot_of_block=slot_of_block, nslots=nslots)


def calib_signatures(N: int, dim: int, ndom: int = 4, seed: int = 0x4B4D):
    """Seeded stand-in for the signatures of N calibration prompts (input construction,
    not the method): each prompt draws a domain; each domain has a nonnegative profile
    (1, or 3 on a random 3/16 of the coordinates); counts are Poisson around 4x the
    profile; each row is scaled to unit L2 norm.  Returns (fp32 [N][dim], domain [N])."""
    rs = np.random.RandomState(seed & 0xFFFFFFFF)
    prof = 1.0 + 2.0 * (rs.random_sample((ndom, dim)) < 3.0 / 16.0)
    dom = rs.randint(0, ndom, size=N)
    counts = rs.poisson(4.0 * prof[dom]).astype(np.float64)
    counts[counts.sum(axis=1) == 0, 0] = 1.0
    sig = counts / np.linalg.norm(counts, axis=1, keepdims=True)
    return sig.astype(np.float32), dom.astype(np.int32)


def kmeans_seed_rows(N: int, D: int, seed: int = 0x5EED) -> np.ndarray:
    """D distinct row indices, the initial centroids of a K-means fit (seeded choice)."""
    return np.random.RandomState(seed & 0xFFFFFFFF).choice(N, size=D, replace=False)
