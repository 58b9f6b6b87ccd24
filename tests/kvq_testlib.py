"""Test helpers: build the same cache through the CUDA library and the oracle,
and compare them (page bytes, window, lengths, dequantized values, attention)."""
from __future__ import annotations

import numpy as np
import torch

import kvq_inputs as W
from oracle import kvq_oracle as O

ATT_TOL = 1e-3  # relative L2 per (sequence, query head), against the oracle on the same dequantized values


def to_c(cfg: O.Config):
    import asymmetric_quantized_kv_gb300 as K
    k, v = cfg.k, cfg.v
    return K.make_config(cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim, (k.fmt, k.mode, k.axis, k.group),
                         (v.fmt, v.mode, v.axis, v.group), cfg.residual, cfg.page_size, cfg.rope_pre,
                         cfg.rope_theta, cfg.src_dtype, cfg.meta_dtype)


def torch_src(x: np.ndarray, cfg: O.Config, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if cfg.src_dtype == O.BF16:
        t = t.to(torch.bfloat16)  # values are bf16-exact already: exact conversion
    return t.to(device)


class Case:
    """Synthetic streams K[b][h], V[b][h] ([T_b, D] float32, exact in the source
    dtype), per-head static scales, a GPU cache filled by chunked appends and
    the oracle states."""

    def __init__(self, cfg: O.Config, lens, seed=0, outliers=(3, 17), factor=30.0, chunking="random",
                 permute_pages=True, extra_pages=1, streams=None, static_scales=None, rope_table=True):
        """rope_table (pre-RoPE keys): True, a table for every position the pages hold;
        False, none (the decode kernel computes the cos/sin); an int n, a table of
        the first n positions only."""
        import asymmetric_quantized_kv_gb300 as K
        self.cfg, self.lens, self.seed = cfg, list(lens), seed
        Bn, H, D, P = len(lens), cfg.num_kv_heads, cfg.head_dim, cfg.page_size
        bf = cfg.src_dtype == O.BF16
        if streams is not None:  # caller-provided K[b][h], V[b][h] ([T_b, D], exact in the source dtype)
            self.K, self.V = streams
        else:
            self.K = [[W.small_stream(seed * 1000 + b * 10 + h, int(lens[b]), D, outliers, factor, bf)
                       for h in range(H)] for b in range(Bn)]
            self.V = [[W.small_stream(seed * 1000 + 500 + b * 10 + h, int(lens[b]), D, (), 1.0, bf)
                       for h in range(H)] for b in range(Bn)]
        # static per-head scales over all sequences (oracle) and through the library
        qk = O.fp8_max(cfg.k.fmt) if O.is_fp8(cfg.k.fmt) else float(O.sym_qmax(O.bits_of(cfg.k.fmt)))
        qv = O.fp8_max(cfg.v.fmt) if O.is_fp8(cfg.v.fmt) else float(O.sym_qmax(O.bits_of(cfg.v.fmt)))
        cat = lambda S, h: np.concatenate([S[b][h] for b in range(Bn)]) if sum(lens) else np.zeros((0, D))
        self.k_scale = [O.calibrate_absmax(cat(self.K, h), qk) for h in range(H)]
        self.v_scale = [O.calibrate_absmax(cat(self.V, h), qv) for h in range(H)]
        self.maxp = max(1, (max(lens) + P - 1) // P + extra_pages)
        n_pages = Bn * self.maxp
        bt = np.arange(n_pages, dtype=np.int32)
        if permute_pages:
            bt = W.page_permutation(n_pages, seed + 17)
        self.block_table = bt.reshape(Bn, self.maxp)
        self.c_cfg = to_c(cfg)
        if cfg.rope_pre and not isinstance(rope_table, bool):
            n = int(rope_table)
            table = torch.empty(K.kvq_rope_table_bytes(self.c_cfg, n), dtype=torch.uint8, device="cuda")
            K.kvq_rope_table_init(self.c_cfg, n, table)
            rope_table = (table, n)
        self.cache = K.PagedKVCache(self.c_cfg, Bn, self.maxp, n_pages, self.block_table, rope_table=rope_table)
        if static_scales is not None:  # given per-head scales (e.g. the uncalibrated unit scale)
            self.k_scale = [float(O.fl32(x)) for x in static_scales[0]]
            self.v_scale = [float(O.fl32(x)) for x in static_scales[1]]
            self.cache.k_scale.copy_(torch.tensor(self.k_scale, dtype=torch.float32))
            self.cache.v_scale.copy_(torch.tensor(self.v_scale, dtype=torch.float32))
        elif sum(lens):
            ks = torch_src(np.concatenate([np.stack([self.K[b][h] for h in range(H)], 1) for b in range(Bn)]), cfg)
            vs = torch_src(np.concatenate([np.stack([self.V[b][h] for h in range(H)], 1) for b in range(Bn)]), cfg)
            self.cache.calibrate(ks, vs, qk, qv)
        self._append_all(chunking)
        self.states = [[O.quantize_stream(cfg, self.K[b][h], self.V[b][h], self.k_scale[h], self.v_scale[h])
                        for h in range(H)] for b in range(Bn)]

    def _append_all(self, chunking):
        cfg = self.cfg
        Bn, H, D = len(self.lens), cfg.num_kv_heads, cfg.head_dim
        g = np.random.default_rng(self.seed + 99)
        done = [0] * Bn
        while any(done[b] < self.lens[b] for b in range(Bn)):
            if chunking == "all":
                take = [self.lens[b] - done[b] for b in range(Bn)]
            elif chunking == "one":
                take = [min(1, self.lens[b] - done[b]) for b in range(Bn)]
            else:
                take = [min(int(g.integers(1, 3 * max(cfg.residual, 16))), self.lens[b] - done[b]) for b in range(Bn)]
            n = max(take)
            kn = np.zeros((Bn, n, H, D), np.float32)
            vn = np.zeros((Bn, n, H, D), np.float32)
            for b in range(Bn):
                for h in range(H):
                    kn[b, :take[b], h] = self.K[b][h][done[b]:done[b] + take[b]]
                    vn[b, :take[b], h] = self.V[b][h][done[b]:done[b] + take[b]]
            per = torch.tensor(take, dtype=torch.int32, device="cuda")
            self.cache.append(torch_src(kn, cfg), torch_src(vn, cfg), per)
            for b in range(Bn):
                done[b] += take[b]
        torch.cuda.synchronize()

    # ---------------------------------------------------------------- comparisons
    def oracle_pages(self):
        L = O.layout(self.cfg)
        n_pages = self.cache.n_pages
        pages = np.zeros((n_pages, L["page"]), np.uint8)
        defined = np.zeros_like(pages, dtype=bool)
        for b in range(len(self.lens)):
            for h in range(self.cfg.num_kv_heads):
                O.write_head_pages(self.cfg, pages, defined, self.block_table, b, h, self.states[b][h])
        return pages, defined

    def check_pages(self):
        pages, defined = self.oracle_pages()
        gpu = self.cache.page_view().cpu().numpy()
        bad = np.nonzero((gpu != pages) & defined)
        assert bad[0].size == 0, f"{bad[0].size} page bytes differ, first at page {bad[0][0]} byte {bad[1][0]}"

    def check_lengths_and_window(self):
        assert self.cache.seq_lens.cpu().tolist() == self.lens
        if self.cfg.residual:
            kw = self.cache.k_win.float().cpu().numpy()
            vw = self.cache.v_win.float().cpu().numpy()
            for b, T in enumerate(self.lens):
                for h in range(self.cfg.num_kv_heads):
                    st = self.states[b][h]
                    r = T - st.n_q
                    assert np.array_equal(kw[b, :r, h], st.k_win.astype(np.float32))
                    assert np.array_equal(vw[b, :r, h], st.v_win.astype(np.float32))

    def check_scales(self):
        ks = self.cache.k_scale.cpu().numpy().astype(np.float64)
        vs = self.cache.v_scale.cpu().numpy().astype(np.float64)
        assert np.array_equal(ks, np.array(self.k_scale)) and np.array_equal(vs, np.array(self.v_scale))

    def check_dequantize(self):
        for b, T in enumerate(self.lens):
            if T == 0:
                continue
            k, v = self.cache.dequantize(b, 0, T)
            k, v = k.cpu().numpy(), v.cpu().numpy()
            for h in range(self.cfg.num_kv_heads):
                ko, vo = O.dequantize_stream(self.cfg, self.states[b][h], self.k_scale[h], self.v_scale[h])
                assert np.array_equal(k[:, h].astype(np.float64), ko), (b, h)
                assert np.array_equal(v[:, h].astype(np.float64), vo), (b, h)

    def queries(self, seed=5):
        g = np.random.default_rng(seed)
        q = g.standard_normal((len(self.lens), self.cfg.num_q_heads, self.cfg.head_dim)).astype(np.float32)
        if self.cfg.src_dtype == O.BF16:
            q = W.bf16_round(q)[1]
        return q

    def check_attention(self, q=None, scale=None, tol=ATT_TOL):
        cfg = self.cfg
        q = self.queries() if q is None else q
        out = self.cache.attention(torch_src(q, cfg), softmax_scale=0.0 if scale is None else scale)
        out = out.cpu().numpy().astype(np.float64)
        worst = 0.0
        for b in range(len(self.lens)):
            for h in range(cfg.num_kv_heads):
                heads = slice(h * cfg.n_rep, (h + 1) * cfg.n_rep)
                ref = O.decode_head(cfg, self.states[b][h], q[b, heads].astype(np.float64), self.k_scale[h],
                                    self.v_scale[h], scale)
                got = out[b, heads]
                if self.lens[b] == 0:
                    assert np.all(got == 0)
                    continue
                err = np.linalg.norm(got - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
                worst = max(worst, float(err.max()))
        assert worst <= tol, f"attention rel L2 {worst:.3e} > {tol}"
        assert int(self.cache.status.item()) == 0
        return worst


class FullCase:
    """A benchmark-sized workload (configs 3, 4, 5 of bench.py) filled through the
    library from seeded device-side draws, exactly as bench.py fills it, with
    host copies of the sampled (sequence, kv-head) source streams.  Static FP8
    scales are fl32(absmax / qmax) (qmax 448 for E4M3, 57344 for E5M2) with the
    absmax taken by torch, so the oracle and the library quantize with the same
    scale without the library computing it."""

    def __init__(self, cid, samples, gen_seed=1, fp8="e4m3", meta="f32", rope_table=True):
        import bench
        import asymmetric_quantized_kv_gb300 as K
        spec = bench.workload_spec(cid, 0, fp8, meta)
        w = spec["w"]
        self.spec, self.w = spec, w
        Bn, H, D, Hq = w.batch, w.num_kv_heads, w.head_dim, w.num_q_heads
        self.lens = [int(x) for x in W.lengths(w)]
        P = spec["P"]
        self.cfg = O.Config(Hq, H, D, O.QSpec(*spec["k"]), O.QSpec(*spec["v"]), spec["R"], P, spec["rope"],
                            spec["theta"], O.BF16, meta_dtype=O.F16 if meta == "f16" else O.F32)
        need = [(T + P - 1) // P for T in self.lens]
        maxp, n_pages = max(need), sum(need)
        perm = W.page_permutation(n_pages, 5)
        bt = np.zeros((Bn, maxp), np.int32)
        o = 0
        for b in range(Bn):
            bt[b, :need[b]] = perm[o:o + need[b]]
            o += need[b]
        self.cache = K.PagedKVCache(to_c(self.cfg), Bn, maxp, n_pages, bt, rope_table=rope_table)
        dev = torch.device("cuda")
        scale = W.torch_outlier_scale(w, dev)
        g = torch.Generator(device=dev)
        g.manual_seed(gen_seed)
        chunk = 4096 if Bn * H * D * 4096 * 2 < (1 << 31) else 1024
        T_max = max(self.lens)
        self.k_scale = [0.0] * H
        self.v_scale = [0.0] * H
        if O.is_fp8(self.cfg.k.fmt):
            qmax = O.fp8_max(self.cfg.k.fmt)
            state = g.get_state()
            kmax = torch.zeros(H, device=dev)
            vmax = torch.zeros(H, device=dev)
            done = 0
            while done < T_max:
                n = min(chunk, T_max - done)
                kk, vv = W.torch_kv_chunk(w, g, Bn, n, scale, dev)
                kmax = torch.maximum(kmax, kk.float().abs().amax(dim=(0, 1, 3)))
                vmax = torch.maximum(vmax, vv.float().abs().amax(dim=(0, 1, 3)))
                done += n
            self.k_scale = [float(O.fl32(a / qmax)) for a in kmax.double().cpu().tolist()]
            self.v_scale = [float(O.fl32(a / qmax)) for a in vmax.double().cpu().tolist()]
            self.cache.k_scale.copy_(torch.tensor(self.k_scale, dtype=torch.float32))
            self.cache.v_scale.copy_(torch.tensor(self.v_scale, dtype=torch.float32))
            g.set_state(state)
        self.keep_all = samples == "all"
        self.samples = [] if self.keep_all else list(samples)
        parts = {s: ([], []) for s in self.samples}
        self.chunks = []  # keep_all: host bf16 copies of every appended chunk
        done = 0
        while done < T_max:
            n = min(chunk, T_max - done)
            take = [max(0, min(n, T - done)) for T in self.lens]
            kk, vv = W.torch_kv_chunk(w, g, Bn, n, scale, dev)
            self.cache.append(kk, vv, torch.tensor(take, dtype=torch.int32, device=dev))
            if self.keep_all:
                self.chunks.append((done, kk.cpu(), vv.cpu()))
            for (b, h) in self.samples:
                if take[b]:
                    parts[(b, h)][0].append(kk[b, :take[b], h].float().cpu().numpy())
                    parts[(b, h)][1].append(vv[b, :take[b], h].float().cpu().numpy())
            done += n
        torch.cuda.synchronize()
        self.streams = {s: (np.concatenate(k), np.concatenate(v)) for s, (k, v) in parts.items()}
        self.q = torch.randn(Bn, Hq, D, generator=g, device=dev).to(torch.bfloat16)

    def source_rows(self, b):
        """keep_all: the source rows of sequence b as float32 [T, Hkv, D] (K, V)."""
        T = self.lens[b]
        ks = [kk[b, :max(0, min(kk.shape[1], T - t0))] for t0, kk, _ in self.chunks if t0 < T]
        vs = [vv[b, :max(0, min(vv.shape[1], T - t0))] for t0, _, vv in self.chunks if t0 < T]
        return torch.cat(ks).float().numpy(), torch.cat(vs).float().numpy()

    def check_every_stream(self, tol=ATT_TOL, workers=16):
        """keep_all: every (sequence, kv-head) stream against the oracle in a
        spawned process pool: kvq_dequantize over the whole stream bit-exact, and
        the attention of the stream's query heads within `tol`.  Returns the
        worst relative L2 and the per-(sequence, query head) errors."""
        import concurrent.futures as cf
        import multiprocessing as mp
        from kvq_oracle_pool import check_stream
        assert self.keep_all
        out = self.cache.attention(self.q).cpu().numpy()
        q = self.q.float().cpu().numpy()
        n_rep, H = self.cfg.n_rep, self.cfg.num_kv_heads
        errs = np.zeros((len(self.lens), self.cfg.num_q_heads))
        bad = []

        def tasks():
            for b, T in enumerate(self.lens):
                K_, V_ = self.source_rows(b)
                kd, vd = self.cache.dequantize(b, 0, T)
                kd, vd = kd.cpu().numpy(), vd.cpu().numpy()
                for h in range(H):
                    heads = slice(h * n_rep, (h + 1) * n_rep)
                    yield ((b, h), self.cfg, K_[:, h], V_[:, h], q[b, heads], kd[:, h], vd[:, h], out[b, heads],
                           self.k_scale[h], self.v_scale[h])

        with cf.ProcessPoolExecutor(workers, mp_context=mp.get_context("spawn")) as ex:
            for (b, h), exact, err in ex.map(check_stream, tasks(), chunksize=1):
                if not exact:
                    bad.append((b, h))
                errs[b, h * n_rep:(h + 1) * n_rep] = err
        assert not bad, f"kvq_dequantize differs from the oracle on streams {bad[:8]}"
        assert errs.max() <= tol, f"attention rel L2 {errs.max():.3e} > {tol}"
        assert int(self.cache.status.item()) == 0
        return float(errs.max()), errs

    def state(self, b, h):
        K_, V_ = self.streams[(b, h)]
        return O.quantize_stream(self.cfg, K_, V_, self.k_scale[h], self.v_scale[h])

    def check_attention(self, tol=ATT_TOL):
        out = self.cache.attention(self.q).cpu().numpy().astype(np.float64)
        q = self.q.float().cpu().numpy().astype(np.float64)
        n_rep = self.cfg.n_rep
        worst = 0.0
        for (b, h) in self.samples:
            heads = slice(h * n_rep, (h + 1) * n_rep)
            ref = O.decode_head(self.cfg, self.state(b, h), q[b, heads], self.k_scale[h], self.v_scale[h])
            err = np.linalg.norm(out[b, heads] - ref, axis=1) / np.linalg.norm(ref, axis=1)
            worst = max(worst, float(err.max()))
        assert worst <= tol, f"attention rel L2 {worst:.3e} > {tol}"
        assert int(self.cache.status.item()) == 0
        return worst

    def check_dequantize(self, span=None):
        """Bit-exact kvq_dequantize against the oracle on each sampled stream: the
        whole stream, or (span given) its first, a middle and its last `span`
        tokens."""
        for (b, h) in self.samples:
            T = self.lens[b]
            ko, vo = O.dequantize_stream(self.cfg, self.state(b, h), self.k_scale[h], self.v_scale[h])
            span_b = T if span is None else span
            for t0 in sorted({0, max(0, T // 2 - span_b // 2), max(0, T - span_b)}):
                t1 = min(T, t0 + span_b)
                k, v = self.cache.dequantize(b, t0, t1)
                assert np.array_equal(k[:, h].cpu().numpy().astype(np.float64), ko[t0:t1]), (b, h, t0)
                assert np.array_equal(v[:, h].cpu().numpy().astype(np.float64), vo[t0:t1]), (b, h, t0)
