// Fused exact-attention forward, one query tile per CTA with a deep S
// pipeline (sm_103a).
//
// Same method as attn_fwd_kernel.cuh (FlashAttention-3 deep-reading report,
// "第三层" intro and §3.1-§3.3: online softmax over key tiles, output rescaled
// when the running maximum moves, divided by the running sum at the end), with
// a different overlap of softmax and GEMMs.  There, P_t(u) overwrites S_t(u),
// so S_t(u+1) can only start after the tile's softmax of step u, and the
// softmax of each tile waits for its own GEMMs every step.  Here S has
// S_BUFS buffers in tensor memory: S(u + S_BUFS) is computed while the
// softmax of S(u) runs, so the softmax of consecutive key tiles runs back to
// back (§3.2's overlap of one iteration's GEMM with the next one's softmax,
// S_BUFS - 1 iterations deep).
//
// Roles (one CTA per SM, 256 threads):
//   warps 0-3   softmax; warp w serves TMEM lanes 32 w .. +31 (one query row
//               per thread)
//   warp 4      TMA producer: Q, then ring stages {K(i), V(i - S_BUFS)}
//   warp 5      MMA issuer: per stage, O += P(i - S_BUFS) V, then
//               S(i) = Q K(i)^T into buffer i % S_BUFS
//   warps 6-7   idle
// Tensor memory: S buffers at columns BN b (b < S_BUFS), P(i) over the first
// columns of its S buffer, O at columns BN S_BUFS .. + D.
//
// The O rescale of step u needs O += P(u-1) V complete; that PV is committed
// to its own barrier, which the softmax waits on before the rescale (it has
// normally completed by then).  Every wait is bounded (see attn_fwd_kernel.cuh).
#pragma once

#include "attn_fwd_kernel.cuh"

namespace attn {

template <int D_, int BN_, bool FP8_, int S_BUFS_, bool SPARSE_ = false>
struct LaCfg : FwdCfg<D_, BN_, 1, FP8_, SPARSE_> {
    using Base = FwdCfg<D_, BN_, 1, FP8_, SPARSE_>;
    static constexpr int S_BUFS = S_BUFS_;      // S buffers in tensor memory
    static constexpr int SOFTMAX_WARPS = 4;
    static constexpr int LOAD_WARP = 4;
    static constexpr int MMA_WARP = 5;
    static constexpr int MMA_WARPS = 1;
    // 256 threads: every warp keeps the launch allocation (no register split).
    static constexpr int THREADS = 256;
    static constexpr int S_STRIDE = BN_;          // TMEM columns per S buffer
    static constexpr int O_COL0 = S_STRIDE * S_BUFS;
    static constexpr int SMEM_BYTES = 1024 + Base::Q_TILE_BYTES + Base::NSTAGE * Base::STAGE_BYTES + Base::BAR_BYTES;
    static_assert(O_COL0 + D_ <= 512, "tensor memory budget");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(S_BUFS >= 2 && S_BUFS <= 4, "S buffers");
    static_assert(BN_ % (FP8_ ? 64 : 32) == 0, "key tile");
};

struct LaBarriers {
    uint64_t q_full, q_empty;
    uint64_t s_full[4], p_full[4];
    uint64_t pv_done, o_full, drain;
    uint64_t ring_full[8], ring_empty[8];
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(LaBarriers) <= 256, "barrier block (FwdCfg::BAR_BYTES)");

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    attn_fwd_la_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_v, const FwdParams p) {
    constexpr int D = Cfg::D, BN = Cfg::BN, BM = Cfg::BM, NSTAGE = Cfg::NSTAGE;
    constexpr int L = Cfg::S_BUFS;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sKV = smem + Cfg::Q_TILE_BYTES;                    // NSTAGE x {K tile, V tile}
    LaBarriers* bars = reinterpret_cast<LaBarriers*>(sKV + NSTAGE * Cfg::STAGE_BYTES);
    volatile int* abort_flag = &bars->abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->q_empty, 1);
        for (int b = 0; b < L; ++b) {
            mbar_init(&bars->s_full[b], 1);
            mbar_init(&bars->p_full[b], Cfg::SOFTMAX_WARPS);   // one arrival per softmax warp
        }
        mbar_init(&bars->pv_done, 1);
        mbar_init(&bars->o_full, 1);
        mbar_init(&bars->drain, 1);
        for (int s = 0; s < 8; ++s) {
            mbar_init(&bars->ring_full[s], 1);
            mbar_init(&bars->ring_empty[s], 1);
        }
        bars->abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == Cfg::LOAD_WARP && lane == 0) {
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
    }
    if (warp == 0) {
        tmem_alloc(&bars->tmem_base, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const int total_items = p.n_mblocks * p.B * p.H;

    if (warp >= Cfg::SOFTMAX_WARPS) {
    if (warp == Cfg::LOAD_WARP) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            uint32_t it = 0, qn = 0;
            bool ok = true;
            for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < total_items && ok; ++rnd) {
                const int item = round_item(rnd);
                if (item >= total_items) continue;
                const WorkItem<1> w = decode_item<Cfg>(p, item);
                if (!w.active[0]) continue;
                const TileKeys tk = tile_keys<Cfg>(w, 0);
                if (!wait_phase(&bars->q_empty, (qn & 1) ^ 1, abort_flag, p, SITE_LOAD_EMPTY)) {
                    ok = false;
                    break;
                }
                ++qn;
                mbar_arrive_expect_tx(&bars->q_full, Cfg::Q_TILE_BYTES);
#pragma unroll
                for (int cb = 0; cb < Cfg::NCB; ++cb)
                    tma_load_4d(sQ + cb * (BM * Cfg::SW), &tmap_q, &bars->q_full, cb * Cfg::BOX_ELEMS, w.h, w.q0,
                                w.b, pol_q);
                // Stage i carries K of the i-th key tile and V of the (i - L)-th.
                int ku = tk.first;
                int hist[L];
#pragma unroll
                for (int x = 0; x < L; ++x) hist[x] = -1;
                while (ok) {
                    const int vkey = hist[L - 1];
                    bool any = ku >= 0;
#pragma unroll
                    for (int x = 0; x < L; ++x) any = any || hist[x] >= 0;
                    if (!any) break;
                    const uint32_t stage = it % NSTAGE, round = it / NSTAGE;
                    if (!wait_phase(&bars->ring_empty[stage], (round & 1) ^ 1, abort_flag, p, SITE_LOAD_EMPTY)) {
                        ok = false;
                        break;
                    }
                    const bool with_k = ku >= 0, with_v = vkey >= 0;
                    mbar_arrive_expect_tx(&bars->ring_full[stage],
                                          (with_k ? Cfg::KV_TILE_BYTES : 0) + (with_v ? Cfg::KV_TILE_BYTES : 0));
                    uint8_t* dst = sKV + stage * Cfg::STAGE_BYTES;
                    if (with_k) {
#pragma unroll
                        for (int cb = 0; cb < Cfg::NCB; ++cb)
                            tma_load_4d(dst + cb * (BN * Cfg::SW), &tmap_k, &bars->ring_full[stage],
                                        cb * Cfg::BOX_ELEMS, w.h / p.group, ku * BN, w.b, pol_kv);
                    }
                    if (with_v) {
#pragma unroll
                        for (int cb = 0; cb < Cfg::NCB; ++cb)
                            tma_load_4d(dst + Cfg::KV_TILE_BYTES + cb * (BN * Cfg::SW), &tmap_v,
                                        &bars->ring_full[stage], cb * Cfg::BOX_ELEMS, w.h / p.group, vkey * BN, w.b,
                                        pol_kv);
                    }
                    ++it;
#pragma unroll
                    for (int x = L - 1; x > 0; --x) hist[x] = hist[x - 1];
                    hist[0] = ku;
                    ku = ku >= 0 ? next_in<Cfg>(tk, ku) : -1;
                }
            }
            const uint32_t first = it > NSTAGE ? it - NSTAGE : 0;
            for (uint32_t k = first; k < it; ++k)
                drain_wait(&bars->ring_full[k % NSTAGE], (k / NSTAGE) & 1, p, SITE_LOAD_DRAIN);
            if (qn > 0) drain_wait(&bars->q_full, (qn - 1) & 1, p, SITE_LOAD_DRAIN);
        }
        __syncwarp();
    } else if (warp == Cfg::MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t sKV_addr = smem_u32(sKV);
        const uint64_t qdesc = sdesc_swz<Cfg::SW>(smem_u32(sQ), 16, 8 * Cfg::SW);
        uint32_t it = 0, qn = 0, s_cnt = 0, pv_cnt = 0;
        bool ok = true;
        for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < total_items && ok; ++rnd) {
            const int item = round_item(rnd);
            if (item >= total_items) continue;
            const WorkItem<1> w = decode_item<Cfg>(p, item);
            if (!w.active[0]) continue;
            const TileKeys tk = tile_keys<Cfg>(w, 0);
            ok = warp_wait(&bars->q_full, qn & 1, abort_flag, p, SITE_MMA_Q);
            ++qn;
            if (!ok) break;
            int ku = tk.first;
            int hist[L];
#pragma unroll
            for (int x = 0; x < L; ++x) hist[x] = -1;
            bool first_pv = true;
            while (true) {
                const int vkey = hist[L - 1];
                bool any = ku >= 0;
#pragma unroll
                for (int x = 0; x < L; ++x) any = any || hist[x] >= 0;
                if (!any) break;
                const uint32_t stage = it % NSTAGE, round = it / NSTAGE;
                ++it;
                if (!warp_wait(&bars->ring_full[stage], round & 1, abort_flag, p, SITE_MMA_FULL)) {
                    ok = false;
                    break;
                }
                const bool do_pv = vkey >= 0, do_s = ku >= 0;
                const uint32_t pb = pv_cnt % L, sb = s_cnt % L;
                if (do_pv && !warp_wait(&bars->p_full[pb], (pv_cnt / L) & 1, abort_flag, p, SITE_MMA_P)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t st_addr = sKV_addr + stage * Cfg::STAGE_BYTES;
                if (elect_one()) {
                    if (do_pv) {
                        const uint64_t vdesc =
                            sdesc_swz<Cfg::SW>(st_addr + Cfg::KV_TILE_BYTES, BN * Cfg::SW, 8 * Cfg::SW);
                        issue_pv<Cfg>(tmem + Cfg::O_COL0, tmem + pb * Cfg::S_STRIDE, vdesc, !first_pv);
                        mma_commit(vkey == tk.last ? &bars->o_full : &bars->pv_done);
                    }
                    if (do_s) {
                        const uint64_t kdesc = sdesc_swz<Cfg::SW>(st_addr, 16, 8 * Cfg::SW);
                        issue_qk<Cfg>(tmem + sb * Cfg::S_STRIDE, qdesc, kdesc);
                        mma_commit(&bars->s_full[sb]);
                        if (ku == tk.last) mma_commit(&bars->q_empty);
                    }
                    if (do_pv || do_s) mma_commit(&bars->ring_empty[stage]);
                    else mbar_arrive(&bars->ring_empty[stage]);
                }
                __syncwarp();
                if (do_pv) {
                    first_pv = false;
                    ++pv_cnt;
                }
                if (do_s) ++s_cnt;
#pragma unroll
                for (int x = L - 1; x > 0; --x) hist[x] = hist[x - 1];
                hist[0] = ku;
                ku = ku >= 0 ? next_in<Cfg>(tk, ku) : -1;
            }
        }
        if (elect_one()) {
            mma_commit(&bars->drain);
            drain_wait(&bars->drain, 0, p, SITE_MMA_DRAIN);
        }
        __syncwarp();
    }
    } else {
        // ------------------------------------------------------------ softmax
        const int r = warp * 32 + lane;           // query row within the tile
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t s_base = tmem + lane_off;  // P(i) goes over the first columns of S(i)
        const uint32_t o_tmem = tmem + lane_off + Cfg::O_COL0;
        const int nblk = (p.N + 127) / 128;
        uint32_t s_cnt = 0, qn = 0, pv_seen = 0;
        bool ok = true;
        for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < total_items && ok; ++rnd) {
            const int item = round_item(rnd);
            if (item >= total_items) continue;
            const WorkItem<1> w = decode_item<Cfg>(p, item);
            const TileKeys tk = tile_keys<Cfg>(w, 0);
            const int bh = w.bh, b = w.b, h = w.h;
            const int qs = w.q0;
            if (!tk.in_n) continue;
            const int i = qs + r;
            __nv_bfloat16* orow =
                reinterpret_cast<__nv_bfloat16*>(p.o) + ((static_cast<size_t>(b) * p.N + i) * p.H + h) * D;
            if (!tk.active) {
                // Block-sparse mask: this query tile sees no key.
                if (i < p.N) {
                    uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
                    for (int x = 0; x < D / 8; ++x) dst[x] = make_uint4(0u, 0u, 0u, 0u);
                    p.lse[static_cast<size_t>(bh) * p.N + i] = -INFINITY;
                }
                continue;
            }
            const int klo = p.window > 0 ? i - p.window + 1 : 0;
            const int khi = p.causal ? min(i, p.N - 1) : p.N - 1;
            float vmax = 1.0f, ivmax = 1.0f;
            float q_mult = p.scale_log2;
            const int bh_kv = b * (p.H / p.group) + h / p.group;
            const size_t sb0 = static_cast<size_t>(bh_kv) * nblk;
            if constexpr (Cfg::FP8) {
                vmax = fp8_vmax(p.v_scale + sb0, nblk);
                ivmax = 1.0f / vmax;
                q_mult *= __ldg(p.q_scale + static_cast<size_t>(bh) * nblk + qs / 128);
            }
            // FP8 factors of the next key tile, loaded one step ahead (bf16:
            // the scale alone).
            float nx_mult = q_mult, nx_lg = 0.0f, nx_inv = 1.0f;
            if constexpr (Cfg::FP8)
                fp8_tile_scales<Cfg>(p, sb0 + (tk.first * BN) / 128, q_mult, ivmax, nx_mult, nx_lg, nx_inv);
            float m = -INFINITY;
            float l = 0.0f;
            bool first_tile = true;
            for (int j = tk.first; j >= 0; j = next_in<Cfg>(tk, j)) {
                const uint32_t sb = s_cnt % L;
                const bool wt = wait_phase(&bars->s_full[sb], (s_cnt / L) & 1, abort_flag, p, SITE_SOFTMAX_S);
                if (!__all_sync(0xffffffffu, wt)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sr[BN];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) tmem_ld32(s_base + sb * Cfg::S_STRIDE + c * 32, sr + c * 32);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) reg_fence32(sr + c * 32);
                const float mult = nx_mult;
                const int kbase = j * BN;
                if (kbase < klo || kbase + BN - 1 > khi) {
#pragma unroll
                    for (int c = 0; c < BN; ++c) {
                        const int key = kbase + c;
                        if (key < klo || key > khi) sr[c] = __float_as_uint(-INFINITY);
                    }
                }
                float mx0 = __uint_as_float(sr[0]), mx1 = __uint_as_float(sr[1]);
                float mx2 = __uint_as_float(sr[2]), mx3 = __uint_as_float(sr[3]);
#pragma unroll
                for (int c = 4; c + 8 <= BN; c += 8) {
                    mx0 = fmax3(mx0, __uint_as_float(sr[c + 0]), __uint_as_float(sr[c + 1]));
                    mx1 = fmax3(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
                    mx2 = fmax3(mx2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
                    mx3 = fmax3(mx3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
                }
                mx0 = fmax3(mx0, mx1, __uint_as_float(sr[BN - 4]));
                mx2 = fmax3(mx2, mx3, __uint_as_float(sr[BN - 3]));
                const float mx = fmax3(mx0, mx2, fmaxf(__uint_as_float(sr[BN - 2]), __uint_as_float(sr[BN - 1])));
                const float m_tile = mx * mult;
                float m_new = m;
                if (m_tile > m + Cfg::RESCALE_LOG2 || m == -INFINITY)
                    m_new = fmaxf(m, m_tile + Cfg::RESCALE_HEADROOM);
                const float m_use = m_new == -INFINITY ? 0.0f : m_new;
                const float alpha = ex2_approx(m - m_use);
                const float2 mult2 = make_float2(mult, mult);
                float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
                const uint32_t p_tm = s_base + sb * Cfg::S_STRIDE;
                if constexpr (!Cfg::FP8) {
                    const float2 neg2 = make_float2(-m_use, -m_use);
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t pk[16];
#pragma unroll
                        for (int x = 0; x < 16; ++x) {
                            const int e = c * 32 + 2 * x;
                            float2 t = __ffma2_rn(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])),
                                                  mult2, neg2);
                            t.x = ex2_approx(t.x);
                            t.y = ex2_approx(t.y);
                            if (x & 1) acc1 = __fadd2_rn(acc1, t);
                            else acc0 = __fadd2_rn(acc0, t);
                            pk[x] = pack_bf16x2(t.x, t.y);
                        }
                        tmem_st16(p_tm + c * 16, pk);
                    }
                } else {
                    // P * pv_mult = exp2(x + log2(pv_mult)): the V block scale
                    // rides in the exponent; the tile's sum is divided by it once.
                    // The exponentials are taken two at a time in f16 (FP16
                    // intermediates of the FP8 path, deep-reading report §3.3):
                    // half the MUFU work, and P is rounded to e4m3 next anyway.
                    // The row sum is kept in four f16x2 partial sums (P * pv_mult
                    // <= 445.7, 16 terms per half: <= 7132 < 65504).
                    const float lg = nx_lg;
                    const float2 negs = make_float2(-m_use + lg, -m_use + lg);
                    uint32_t hs0 = 0u, hs1 = 0u, hs2 = 0u, hs3 = 0u;
#pragma unroll
                    for (int c = 0; c < BN / 64; ++c) {
                        uint32_t pk[16];
#pragma unroll
                        for (int x = 0; x < 16; ++x) {
                            const int e = c * 64 + 4 * x;
                            const float2 t0 = __ffma2_rn(
                                make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), mult2, negs);
                            const float2 t1 = __ffma2_rn(
                                make_float2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), mult2, negs);
                            const uint32_t p01 = ex2_f16x2(pack_f16x2(t0.x, t0.y));
                            const uint32_t p23 = ex2_f16x2(pack_f16x2(t1.x, t1.y));
                            if (x & 1) {
                                hs2 = add_f16x2(hs2, p01);
                                hs3 = add_f16x2(hs3, p23);
                            } else {
                                hs0 = add_f16x2(hs0, p01);
                                hs1 = add_f16x2(hs1, p23);
                            }
                            pk[x] = pack_e4m3x4_f16(p01, p23);
                        }
                        tmem_st16(p_tm + c * 16, pk);
                    }
                    acc0 = __fadd2_rn(f16x2_to_float2(hs0), f16x2_to_float2(hs2));
                    acc1 = __fadd2_rn(f16x2_to_float2(hs1), f16x2_to_float2(hs3));
                    const float inv = nx_inv;
                    acc0.x *= inv; acc0.y *= inv; acc1.x *= inv; acc1.y *= inv;
                }
                const float rsum = (acc0.x + acc0.y) + (acc1.x + acc1.y);
                l = l * alpha + rsum;
                if (!first_tile) {
                    // O += P(previous) V must be complete before O is rescaled
                    // (and before the next P V, which follows this arrival).
                    const bool wp = wait_phase(&bars->pv_done, pv_seen & 1, abort_flag, p, SITE_SOFTMAX_O);
                    ++pv_seen;
                    tc_fence_after();
                    if (__all_sync(0xffffffffu, wp) && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t orr[32];
                            tmem_ld32(o_tmem + c * 32, orr);
                            tmem_wait_ld();
                            reg_fence32(orr);
#pragma unroll
                            for (int x = 0; x < 32; ++x)
                                orr[x] = __float_as_uint(__uint_as_float(orr[x]) * alpha);
                            tmem_st32(o_tmem + c * 32, orr);
                        }
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->p_full[sb]);
                if constexpr (Cfg::FP8) {
                    const int jn = next_in<Cfg>(tk, j);
                    if (jn >= 0) {
                        fp8_tile_scales<Cfg>(p, sb0 + (jn * BN) / 128, q_mult, ivmax, nx_mult, nx_lg, nx_inv);
                        pin3(nx_mult, nx_lg, nx_inv);
                    }
                }
                m = m_new;
                first_tile = false;
                ++s_cnt;
            }
            if (!ok) break;
            bool wt = wait_phase(&bars->o_full, qn & 1, abort_flag, p, SITE_SOFTMAX_O);
            ++qn;
            ok = __all_sync(0xffffffffu, wt);
            if (!ok) break;
            tc_fence_after();
            // l = 0 only for a row that sees no key: O = 0, LSE = -inf.
            float out_mult = l > 0.0f ? 1.0f / l : 0.0f;
            if constexpr (Cfg::FP8) out_mult *= vmax * (1.0f / Cfg::P8_SCALE);
            const bool store = i < p.N;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t orr[32];
                tmem_ld32(o_tmem + c * 32, orr);
                tmem_wait_ld();
                reg_fence32(orr);
                uint32_t pk[16];
#pragma unroll
                for (int x = 0; x < 16; ++x)
                    pk[x] = pack_bf16x2(__uint_as_float(orr[2 * x]) * out_mult,
                                        __uint_as_float(orr[2 * x + 1]) * out_mult);
                if (store) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
                    for (int x = 0; x < 4; ++x) dst[x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
                }
            }
            if (store) p.lse[static_cast<size_t>(bh) * p.N + i] = (m + __log2f(l)) * 0.69314718055994530942f;
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

template <class Cfg>
cudaError_t launch_fwd_la(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const FwdParams& p,
                          int max_ctas, cudaStream_t stream) {
    auto kernel = attn_fwd_la_kernel<Cfg>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long units = static_cast<long long>(p.n_mblocks) * p.B * p.H;
    const long long grid = units < max_ctas ? units : max_ctas;
    kernel<<<dim3(static_cast<unsigned>(grid)), dim3(Cfg::THREADS), Cfg::SMEM_BYTES, stream>>>(q, k, v, p);
    return cudaGetLastError();
}

}  // namespace attn
