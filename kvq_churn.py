"""Churn workload with integrity tags, driven through the public binding.

32 layers x 64 requests, GQA 32/8, head_dim 128, page size 16, contexts
U{2,048..65,536}.  A host-side page allocator gives every physical page a
uint32 tag that is bumped each time the page is handed to a new owner; each
request records the tag it expects for each of its pages.  Per step:

  1. 0.5 % of the used block-table entries are seeded to point at a page
     whose tag moved on (the request still expects the old tag), laid down
     as runs inside a few requests so that most requests stay live;
  2. kvq_tag_check once for the step (page ids and tags are shared by the
     layers) -> per-request abort flags;
  3. for every layer: kvq_append of each request's new token (aborted
     requests skipped), then kvq_decode_attn (aborted requests -> zeros);
  4. aborted requests and 20 % of the others finish; their pages go back to
     the pool; new requests take pages from it (tags bumped).

The page contents of every layer start as seeded bf16 values quantised with
kvq_append and are then overwritten by the appended tokens, whose bf16 rows
are seeded per (layer, step).  A checker can therefore rebuild any page's
bf16 contents from the seed and the append log, without reading anything
the CUDA path produced.  This is the pages' integrity layer (blog post
"Smaller, faster, safer", page-2 mirror section "KV Cache 完整性检查";
page-3 mirror section "一个不能出错的共享缓存").
"""
from __future__ import annotations

import math

import numpy as np

import workloads as W

PAGES_PER_CHUNK = 8192          # initial contents are generated per chunk of pages


class PagePool:
    """Host allocator: free list in random order, tag bumped on every reuse."""

    def __init__(self, num_pages: int, rng: np.random.Generator):
        self.num_pages = num_pages
        self.rng = rng
        self.tags = rng.integers(0, 2**32, size=num_pages, dtype=np.uint64).astype(np.uint32)
        self.free = list(rng.permutation(num_pages))
        self.ever_used = np.zeros(num_pages, bool)

    def take(self, n: int):
        if n > len(self.free):
            return None
        pages = [int(self.free.pop()) for _ in range(n)]
        for p in pages:
            if self.ever_used[p]:
                self.tags[p] += np.uint32(1)          # new owner: the tag changes
            self.ever_used[p] = True
        return pages

    def give_back(self, pages):
        self.free.extend(pages)
        order = self.rng.permutation(len(self.free))
        self.free = [self.free[i] for i in order]


class Request:
    def __init__(self, rid: int, length: int, pages, tags):
        self.rid = rid
        self.length = length                  # tokens attended at the next step (incl. its append)
        self.pages = list(pages)
        self.expected = [int(t) for t in tags]


class ChurnState:
    """Host bookkeeping of the churn workload (no GPU, no method arithmetic)."""

    def __init__(self, seed: int = 0, batch: int = 64, page_size: int = 16, lo: int = 2048,
                 hi: int = 65536, steps: int = W.CHURN_STEPS, stale_frac: float = 0.005,
                 finish_frac: float = 0.2, pool_factor: float = 1.2):
        self.rng = np.random.default_rng(seed)
        self.batch, self.ps, self.lo, self.hi = batch, page_size, lo, hi
        self.steps, self.stale_frac, self.finish_frac = steps, stale_frac, finish_frac
        lens = self.rng.integers(lo, hi + 1, size=batch)
        demand = sum(math.ceil((int(L) + steps) / page_size) for L in lens)
        self.num_pages = int(math.ceil(pool_factor * demand))
        self.max_pages = math.ceil((hi + steps) / page_size)
        self.pool = PagePool(self.num_pages, self.rng)
        self.next_rid = 0
        self.slots = [self._new_request(int(L)) for L in lens]
        self.step_index = 0

    def _new_request(self, context: int):
        n = math.ceil((context + 1) / self.ps)
        pages = self.pool.take(n)
        if pages is None:
            return None
        r = Request(self.next_rid, context + 1, pages, self.pool.tags[pages])
        self.next_rid += 1
        return r

    def tables(self):
        """block_table, expected_tags, seq_lens for this step with the seeded
        stale entries, and the set of requests that must be flagged."""
        B, maxp = self.batch, self.max_pages
        bt = np.full((B, maxp), -1, np.int32)
        exp = np.zeros((B, maxp), np.uint32)
        seq = np.zeros(B, np.int32)
        used = 0
        for i, r in enumerate(self.slots):
            if r is None:
                continue
            n = math.ceil(r.length / self.ps)
            bt[i, :n] = r.pages[:n]
            exp[i, :n] = r.expected[:n]
            seq[i] = r.length
            used += n
        # 0.5 % of the used entries go stale, laid down as runs inside a few
        # requests (a request that kept pointers to pages since handed to
        # another owner): the count is the stated fraction, most requests live
        stale = set()
        target = int(round(self.stale_frac * used))
        live = [i for i, r in enumerate(self.slots) if r is not None]
        order = [int(x) for x in self.rng.permutation(live)]
        while target > 0 and order:
            i = order.pop()
            n = math.ceil(int(seq[i]) / self.ps)
            start = int(self.rng.integers(n))
            run = min(n - start, target)
            exp[i, start:start + run] = self.pool.tags[bt[i, start:start + run]] - np.uint32(1)
            target -= run
            stale.add(i)
        return bt, exp, seq, stale

    def advance(self, aborted):
        """Finish the aborted requests and a random 20 % of the rest; admit new ones."""
        live = [i for i, r in enumerate(self.slots) if r is not None]
        keep = [i for i in live if i not in aborted]
        n_finish = int(round(self.finish_frac * len(keep)))
        finish = set(int(i) for i in aborted) | set(
            int(x) for x in self.rng.choice(keep, size=n_finish, replace=False))
        for i in sorted(finish):
            if self.slots[i] is not None:
                self.pool.give_back(self.slots[i].pages)
                self.slots[i] = None
        for i, r in enumerate(self.slots):
            if r is None:
                continue
            r.length += 1
            if math.ceil(r.length / self.ps) > len(r.pages):
                p = self.pool.take(1)
                if p is None:                    # pool exhausted: the request finishes
                    self.pool.give_back(r.pages)
                    self.slots[i] = None
                    continue
                r.pages.extend(p)
                r.expected.append(int(self.pool.tags[p[0]]))
        for i in range(self.batch):
            if self.slots[i] is None:
                self.slots[i] = self._new_request(int(self.rng.integers(self.lo, self.hi + 1)))
        self.step_index += 1


class ChurnDevice:
    """The churn workload's caches (one K and one V cache per layer) in HBM and
    the per-step kernel sequence."""

    def __init__(self, state: ChurnState, layers: int = 32, num_q_heads: int = 32,
                 num_kv_heads: int = 8, seed: int = 0, device: str = "cuda", log_layers=(0,)):
        import torch
        import fp8_quantised_paged_kv_gb300 as kvq
        self.torch, self.kvq = torch, kvq
        self.s, self.layers, self.seed, self.device = state, layers, seed, device
        self.hq, self.hkv, self.D = num_q_heads, num_kv_heads, 128
        self.sigma = 1.0 / math.sqrt(self.D)
        N, ps = state.num_pages, state.ps
        self.desc = kvq.CacheDesc(N, ps, num_kv_heads, self.D, kvq.KVQ_CACHE_FP8_E4M3)
        shape = (N, num_kv_heads, ps, self.D)
        self.k = [torch.empty(shape, dtype=torch.uint8, device=device) for _ in range(layers)]
        self.v = [torch.empty(shape, dtype=torch.uint8, device=device) for _ in range(layers)]
        self.k_scale_host, self.v_scale_host, self.k_scale, self.v_scale = [], [], [], []
        self.log_layers = set(log_layers)
        self.append_log = {l: {} for l in self.log_layers}     # slot -> (k row, v row) bf16 bits
        for l in range(layers):
            self._populate(l)
        self.ws = kvq.workspace_for(self.desc, state.batch, num_q_heads, state.max_pages, 0, device)
        self.abort = torch.zeros(state.batch, dtype=torch.uint8, device=device)

    # ------------------------------------------------------------ values
    def _gen(self, *key):
        from kvq_harness import _gen
        return _gen(self.device, self.seed, *key)

    def initial_chunk(self, layer: int, chunk: int):
        """bf16 K, V of the pages of one chunk, token-major [pages*ps][Hkv][D]."""
        N, ps = self.s.num_pages, self.s.ps
        n = min(PAGES_PER_CHUNK, N - chunk * PAGES_PER_CHUNK)
        g = self._gen(layer, 7, chunk)
        shape = (n * ps, self.hkv, self.D)
        return W.normal_bf16_torch(shape, g, self.device), W.normal_bf16_torch(shape, g, self.device)

    def step_values(self, layer: int, step: int):
        B = self.s.batch
        g = self._gen(layer, 11, step)
        q = W.normal_bf16_torch((B, self.hq, self.D), g, self.device)
        kn = W.normal_bf16_torch((B, self.hkv, self.D), g, self.device)
        vn = W.normal_bf16_torch((B, self.hkv, self.D), g, self.device)
        return q, kn, vn

    def _populate(self, layer: int):
        torch, kvq = self.torch, self.kvq
        N, ps = self.s.num_pages, self.s.ps
        chunks = math.ceil(N / PAGES_PER_CHUNK)
        kmax = torch.zeros(self.hkv, dtype=torch.float32, device=self.device)
        vmax = torch.zeros_like(kmax)
        for c in range(chunks):
            kb, vb = self.initial_chunk(layer, c)
            kmax = torch.maximum(kmax, kb.abs().float().amax(dim=(0, 2)))
            vmax = torch.maximum(vmax, vb.abs().float().amax(dim=(0, 2)))
        ks = W.scales_from_amax(kmax.cpu().numpy())
        vs = W.scales_from_amax(vmax.cpu().numpy())
        self.k_scale_host.append(ks)
        self.v_scale_host.append(vs)
        self.k_scale.append(torch.from_numpy(ks).to(self.device))
        self.v_scale.append(torch.from_numpy(vs).to(self.device))
        for c in range(chunks):
            kb, vb = self.initial_chunk(layer, c)
            first = c * PAGES_PER_CHUNK * ps
            slots = torch.arange(first, first + kb.shape[0], dtype=torch.int64, device=self.device)
            kvq.kvq_append(self.desc, kb, vb, slots, self.k_scale[layer], self.v_scale[layer],
                           None, self.k[layer], self.v[layer])

    # -------------------------------------------------------------- step
    def upload(self, bt, exp, seq):
        torch, s, dev = self.torch, self.s, self.device
        slots = np.full(s.batch, -1, np.int64)
        for i, L in enumerate(seq):
            if L > 0:
                slots[i] = int(bt[i, (L - 1) // s.ps]) * s.ps + (L - 1) % s.ps
        return (torch.from_numpy(bt).to(dev), torch.from_numpy(exp.view(np.int32)).to(dev),
                torch.from_numpy(seq).to(dev), torch.from_numpy(s.pool.tags.view(np.int32)).to(dev),
                slots, torch.from_numpy(slots).to(dev))

    def run_step(self, keep_layers=(), stream=None):
        """One decode step over all layers.  Returns the host tables, the
        seeded stale set, the appended slots, the abort flags (host) and
        {layer: (out, q, k_new, v_new)} for keep_layers."""
        torch, kvq, s = self.torch, self.kvq, self.s
        bt, exp, seq, stale = s.tables()
        bt_d, exp_d, seq_d, tags_d, slots, slots_d = self.upload(bt, exp, seq)
        kvq.kvq_tag_check(bt_d, exp_d, seq_d, s.ps, tags_d, self.abort, stream)
        kept = {}
        for l in range(self.layers):
            q, kn, vn = self.step_values(l, s.step_index)
            kvq.kvq_append(self.desc, kn, vn, slots_d, self.k_scale[l], self.v_scale[l], self.abort,
                           self.k[l], self.v[l], stream)
            out = torch.empty((s.batch, self.hq, self.D), dtype=torch.bfloat16, device=self.device)
            kvq.kvq_decode_attn(self.desc, q, self.k[l], self.v[l], self.k_scale[l], self.v_scale[l],
                                bt_d, seq_d, self.sigma, self.abort, out, self.ws, 0, stream)
            if l in keep_layers or l in self.log_layers:
                kept[l] = (out, q, kn, vn)
        abort = self.abort.cpu().numpy()
        for l in self.log_layers:                  # bf16 rows the oracle needs later
            kn, vn = kept[l][2], kept[l][3]
            knh = kn.view(torch.int16).cpu().numpy().view(np.uint16)
            vnh = vn.view(torch.int16).cpu().numpy().view(np.uint16)
            for i in range(s.batch):
                if slots[i] >= 0 and not abort[i]:
                    self.append_log[l][int(slots[i])] = (knh[i].copy(), vnh[i].copy())
        return bt, exp, seq, stale, slots, abort, kept

    # ------------------------------------------------------ oracle feed
    def request_bf16(self, layer: int, bt_row, length: int):
        """bf16 bits [L][Hkv][D] of K and V of a request's tokens, rebuilt from
        the seeded initial contents and the append log (nothing read back)."""
        torch = self.torch
        ps = self.s.ps
        n_pages = math.ceil(length / ps)
        pages = [int(p) for p in bt_row[:n_pages]]
        k = np.empty((n_pages * ps, self.hkv, self.D), np.uint16)
        v = np.empty_like(k)
        by_chunk = {}
        for i, p in enumerate(pages):
            by_chunk.setdefault(p // PAGES_PER_CHUNK, []).append((i, p))
        for c, items in by_chunk.items():
            kb, vb = self.initial_chunk(layer, c)
            idx = torch.tensor([(p - c * PAGES_PER_CHUNK) * ps + o for _, p in items for o in range(ps)],
                               device=self.device)
            ksel = kb.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
            vsel = vb.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
            for j, (i, _) in enumerate(items):
                k[i * ps:(i + 1) * ps] = ksel[j * ps:(j + 1) * ps]
                v[i * ps:(i + 1) * ps] = vsel[j * ps:(j + 1) * ps]
        log = self.append_log[layer]
        for i, p in enumerate(pages):
            for o in range(ps):
                hit = log.get(p * ps + o)
                if hit is not None:
                    k[i * ps + o], v[i * ps + o] = hit
        return k[:length], v[:length]


class ChurnGraphStep:
    """The churn step (one tag check, then append + decode attention for every
    layer) over fixed device buffers, so that it can be captured once as a
    CUDA graph and replayed each step after the step's tables and values are
    copied in."""

    def __init__(self, dev: ChurnDevice, fused_append: bool = False):
        torch = dev.torch
        self.dev, s = dev, dev.s
        self.fused_append = fused_append      # append inside each layer's decode launch
        B, maxp, d = s.batch, s.max_pages, dev.device
        self.bt = torch.empty((B, maxp), dtype=torch.int32, device=d)
        self.exp = torch.empty((B, maxp), dtype=torch.int32, device=d)
        self.seq = torch.empty(B, dtype=torch.int32, device=d)
        self.tags = torch.empty(s.num_pages, dtype=torch.int32, device=d)
        self.slots = torch.empty(B, dtype=torch.int64, device=d)
        shape_q, shape_kv = (B, dev.hq, dev.D), (B, dev.hkv, dev.D)
        self.q = [torch.empty(shape_q, dtype=torch.bfloat16, device=d) for _ in range(dev.layers)]
        self.kn = [torch.empty(shape_kv, dtype=torch.bfloat16, device=d) for _ in range(dev.layers)]
        self.vn = [torch.empty(shape_kv, dtype=torch.bfloat16, device=d) for _ in range(dev.layers)]
        self.out = [torch.empty(shape_q, dtype=torch.bfloat16, device=d) for _ in range(dev.layers)]
        self.graph = None

    INPUTS = ("bt", "exp", "seq", "tags", "slots")

    def pack_inputs(self):
        """Re-home every per-step input (tables, tags, slots and each layer's q,
        new K and new V) in one device buffer of 256-byte-aligned segments,
        and return it with a pinned host buffer of the same size, so that a
        step fed from host memory is one host-to-device copy."""
        torch, dev = self.dev.torch, self.dev
        tensors = [(n, None) for n in self.INPUTS] + \
            [(n, l) for n in ("q", "kn", "vn") for l in range(dev.layers)]
        get = lambda n, l: getattr(self, n) if l is None else getattr(self, n)[l]
        offs, total = [], 0
        for n, l in tensors:
            t = get(n, l)
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.zeros(total, dtype=torch.uint8, device=dev.device)
        for (n, l), o in zip(tensors, offs):
            t = get(n, l)
            view = buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
            if l is None:
                setattr(self, n, view)
            else:
                getattr(self, n)[l] = view
        self.packed = buf
        self.packed_host = torch.zeros(total, dtype=torch.uint8).pin_memory()
        return self.packed_host, self.packed

    def load(self):
        """Copy this step's tables and per-layer values into the fixed buffers.
        Returns (bt, exp, seq, stale, slots) on the host."""
        dev, s = self.dev, self.dev.s
        bt, exp, seq, stale = s.tables()
        bt_d, exp_d, seq_d, tags_d, slots, slots_d = dev.upload(bt, exp, seq)
        self.bt.copy_(bt_d)
        self.exp.copy_(exp_d)
        self.seq.copy_(seq_d)
        self.tags.copy_(tags_d)
        self.slots.copy_(slots_d)
        for l in range(dev.layers):
            q, kn, vn = dev.step_values(l, s.step_index)
            self.q[l].copy_(q)
            self.kn[l].copy_(kn)
            self.vn[l].copy_(vn)
        return bt, exp, seq, stale, slots

    def pack_outputs(self):
        """Every layer's output as a view of one [layers][B][Hq][D] tensor (one
        device-to-host copy reads them all); returns that tensor."""
        torch, dev = self.dev.torch, self.dev
        allout = torch.empty((dev.layers,) + tuple(self.out[0].shape), dtype=self.out[0].dtype,
                             device=dev.device)
        self.out = [allout[l] for l in range(dev.layers)]
        return allout

    def launch(self, stream=None, after_check=None, layer_events=None):
        """The step's launches: the tag check, then every layer.  Optional
        CUDA events: `after_check` is recorded between the check and the first
        layer, layer_events[l] = (start, end) around layer l's decode launch."""
        dev, kvq, s = self.dev, self.dev.kvq, self.dev.s
        kvq.kvq_tag_check(self.bt, self.exp, self.seq, s.ps, self.tags, dev.abort, stream)
        if after_check is not None:
            after_check.record(stream)
        for l in range(dev.layers):
            if layer_events is not None and self.fused_append:
                layer_events[l][0].record(stream)
            if self.fused_append:
                kvq.kvq_decode_attn_append(dev.desc, self.q[l], dev.k[l], dev.v[l], dev.k_scale[l],
                                           dev.v_scale[l], self.bt, self.seq, dev.sigma, dev.abort,
                                           self.kn[l], self.vn[l], self.out[l], dev.ws, 0, stream)
                if layer_events is not None:
                    layer_events[l][1].record(stream)
                continue
            kvq.kvq_append(dev.desc, self.kn[l], self.vn[l], self.slots, dev.k_scale[l], dev.v_scale[l],
                           dev.abort, dev.k[l], dev.v[l], stream)
            if layer_events is not None:
                layer_events[l][0].record(stream)
            kvq.kvq_decode_attn(dev.desc, self.q[l], dev.k[l], dev.v[l], dev.k_scale[l], dev.v_scale[l],
                                self.bt, self.seq, dev.sigma, dev.abort, self.out[l], dev.ws, 0, stream)
            if layer_events is not None:
                layer_events[l][1].record(stream)

    def capture(self):
        """Capture launch() as a CUDA graph (after one eager launch has run
        every first-call setup of the library)."""
        torch = self.dev.torch
        side = torch.cuda.Stream(device=self.dev.device)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.launch(side)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.launch(torch.cuda.current_stream())
        torch.cuda.synchronize()

    def replay(self):
        self.graph.replay()
