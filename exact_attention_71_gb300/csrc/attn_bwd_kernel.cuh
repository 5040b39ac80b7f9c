// Fused exact-attention backward for sm_103a (bf16, head_dim 64 and 128).
//
// Method (FlashAttention-3 deep-reading report §3.4: the backward keeps
// FA2's recompute strategy, five matrix products against the forward's
// two).  With dO = dL/dO, the forward's O and LSE, and D_i = dO_i . O_i
// (computed beforehand), every (key tile, query tile) pair recomputes
//     P  = exp(scale Q K^T - LSE)          dP = dO V^T
//     dS = P * (dP - D)                    (elementwise)
// and contributes dV += P^T dO, dK += scale dS^T Q, dQ += scale dS K.
//
// GB300 mapping: one CTA per (batch, key/value head, 128-key tile), K and V
// of the tile resident in shared memory for the CTA's lifetime, dK and dV
// accumulated in tensor memory; the CTA walks the 64-row query tiles of
// every query head of the group.  The products are computed transposed so
// that every accumulator has its 128 rows on the tensor-memory lanes:
//     S^T  = K Q^T      (M = 128 keys,  N = 64 queries, K = d)
//     dP^T = V dO^T     (M = 128 keys,  N = 64 queries, K = d)
//     dV  += P^T dO     (A = P^T from tensor memory, B = dO MN-major)
//     dK  += dS^T Q     (A = dS^T from shared memory, B = Q MN-major)
//     dQ^T = K^T dS^T   (A = K read MN-major, B = dS^T from shared memory)
// and dQ^T (128 dims x 64 queries) is added into a float32 accumulator in
// global memory with one bulk reduction per step (other key tiles add into
// the same rows).
//
// Roles (448 threads; 512 at d = 64):
//   warps 0-7   two elementwise warpgroups: thread = key row; P, dS, each
//               for half of the step's query columns
//   warps 8-11  dQ warpgroup: thread = head dimension; dQ^T out of tensor
//               memory into a staging buffer and a bulk add to global
//               memory; at the end the dK epilogue (thread = key row)
//   warp  12    TMA producer: K, V once; per step Q, dO (ring), LSE, D
//   warp  13    MMA issuer (one elected lane)
//   warps 14-15 (d = 64) idle: they complete the fourth warpgroup, so that
//               a register split (setmaxnreg) can raise the elementwise
//               warpgroups above the 128 registers of the launch
// Tensor memory (512 columns, d = 128): dV [0, d), dK [d, 2d), S^T
// double-buffered at 2d and 2d + 64, dP^T at 2d + 128, dQ^T at 2d + 192.
// P (bf16 pairs) overwrites the first columns of its S^T buffer.  dS^T goes to shared
// memory only (double-buffered), where it serves as the K-major A operand of
// dK and the MN-major B operand of dQ^T; so dP^T of the next step can be
// issued as soon as this step's dS is written, ahead of dK and dQ^T, and the
// elementwise warps compute the next dS while the pipe runs them.
// Issue order of step t: dV(t), S(t+1), dP(t+1), dK(t), dQ^T(t).
//
// Every barrier wait is bounded (the forward kernel's failure protocol):
// a role that gives up records a site code, raises the shared abort flag and
// leaves its loop; the CTA's own copies and MMAs are drained before tensor
// memory is freed.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_bulk.cuh"
#include "sm103_ptx.cuh"

namespace attn {

struct BwdParams {
    const float* lse2;     // (B, H, N_pad): LSE * log2(e); +inf in the pad rows
    const float* dvec;     // (B, H, N_pad): D = rowsum(dO * O); 0 in the pad rows
    float* dq_acc;         // (B, H, N_pad, d) float32, zero before the launch
    void* dk;              // bf16 (B, N, H_kv, d)
    void* dv;              // bf16 (B, N, H_kv, d)
    int B, H, H_kv, N, N_pad, group;
    int causal, window;
    float scale;           // softmax scale
    float scale_log2;      // scale * log2(e)
    int n_kblocks;         // ceil(N / 128)
    unsigned long long wait_limit;
    int* status;
};

enum : int {
    BSITE_LOAD_EMPTY = 0x51,
    BSITE_LOAD_DRAIN = 0x52,
    BSITE_MMA_KV = 0x61,
    BSITE_MMA_Q = 0x62,
    BSITE_MMA_P = 0x63,
    BSITE_MMA_DS = 0x64,
    BSITE_MMA_DQ = 0x65,
    BSITE_MMA_DRAIN = 0x66,
    BSITE_EW_S = 0x71,
    BSITE_EW_Q = 0x72,
    BSITE_EW_DP = 0x73,
    BSITE_EW_ACC = 0x74,
    BSITE_DQ_FULL = 0x81,
    BSITE_DQ_ACC = 0x82,
};

template <int D_>
struct BwdCfg {
    static constexpr int D = D_;
    // d = 128: 64 query rows per step, S^T double-buffered, dQ computed
    // transposed (dQ^T = K^T dS^T, head dimensions on the TMEM lanes).
    // d = 64: 128 query rows per step (full-rate N = 128 products), one S^T
    // buffer, dQ = dS K with the queries on the lanes (an M = 64 product is
    // avoided).
    static constexpr bool DQ_T = D == 128;
    static constexpr int BM = D == 128 ? 64 : 128;        // query rows per step
    static constexpr int S_BUFS = D == 128 ? 2 : 1;
    static constexpr int BN = 128;                        // keys per CTA
    static constexpr int NCB = D * 2 / 128;               // 128-byte column boxes per row
    static constexpr int Q_TILE = BM * D * 2;
    static constexpr int KV_TILE = BN * D * 2;
    static constexpr int NST = 2;                         // Q / dO ring depth
    static constexpr int STAGE = 2 * Q_TILE;              // Q, dO
    // dS^T (x2 buffers): rows = keys, BM queries each, in 128-byte column
    // chunks of 64 queries ([chunk][key][64 queries], 128-byte swizzle).
    static constexpr int DS_BYTES = BN * BM * 2;
    static constexpr int DS_CHUNK = BN * 128;             // bytes of one 64-query chunk
    // float32 dQ staging: d = 128, [query][dim] for one bulk add per step
    // (x2 buffers); d = 64, one row per thread padded by 16 bytes (fewer bank
    // conflicts), one bulk add per row.
    static constexpr int DQ_ROW = DQ_T ? D * 4 : D * 4 + 16;
    static constexpr int DQ_STAGE = BM * DQ_ROW;
    static constexpr int DQ_BUFS = DQ_T ? 2 : 1;
    static constexpr int VEC_BYTES = 2 * BM * 4;          // LSE2 and D of one step
    static constexpr int DV_COL = 0, DK_COL = D, S_COL = 2 * D, DP_COL = 2 * D + S_BUFS * BM,
                         DQ_COL = 2 * D + (S_BUFS + 1) * BM;
    static constexpr int DQ_COLS = DQ_T ? BM : D;         // TMEM columns of dQ^T / dQ
    static constexpr int TMEM_COLS = 512;
    // Two elementwise warpgroups, each owning half of the step's query columns.
    static constexpr int EW_WGS = 2, EW_COLS = BM / EW_WGS;
    static constexpr int EW_WARP0 = 0, DQ_WARP0 = 4 * EW_WGS, LOAD_WARP = DQ_WARP0 + 4, MMA_WARP = LOAD_WARP + 1;
    // d = 64: two idle warps complete the load / MMA warpgroup (512 threads,
    // four whole warpgroups), so that a register split can give the
    // elementwise warpgroups, which keep 64 scores of P per thread, more than
    // the 128 registers a thread gets at launch.  d = 128 needs no split.
    static constexpr bool REG_SPLIT = D == 64;
    static constexpr int THREADS = REG_SPLIT ? 512 : (MMA_WARP + 1) * 32;
    static constexpr int LAUNCH_REGS = 128;
    static constexpr int EW_REGS = 152, DQ_REGS = 120, LM_REGS = 88;
    static_assert(!REG_SPLIT || 2 * 128 * EW_REGS + 128 * DQ_REGS + 128 * LM_REGS <= LAUNCH_REGS * THREADS,
                  "register split");
    static constexpr int BAR_BYTES = 256;
    // Shared memory (offsets from a 1024-byte aligned base).
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + KV_TILE;
    static constexpr int OFF_STAGE = OFF_V + KV_TILE;
    static constexpr int OFF_DS = OFF_STAGE + NST * STAGE;
    static constexpr int OFF_DQ = OFF_DS + 2 * DS_BYTES;
    static constexpr int OFF_VEC = OFF_DQ + DQ_BUFS * DQ_STAGE;
    static constexpr int OFF_BAR = OFF_VEC + NST * VEC_BYTES;
    static constexpr int SMEM_BYTES = 1024 + OFF_BAR + BAR_BYTES;

    static_assert(D == 128 || D == 64, "the backward is built for head_dim 64 and 128");
    static_assert(DQ_COL + DQ_COLS <= TMEM_COLS, "tensor memory budget");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

struct BwdBarriers {
    uint64_t kv_full;
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t dp_full;
    uint64_t ds_full;
    uint64_t dq_full;
    uint64_t dq_empty;
    uint64_t acc_full;
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, const BwdParams& p,
                                      int site) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (static_cast<unsigned long long>(clock64() - t0) > p.wait_limit) {
            *abort_flag = 1;
            atomicCAS(p.status, 0, site);
            return false;
        }
    }
}

__device__ __forceinline__ bool bwait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                           const BwdParams& p, int site) {
    return __all_sync(0xffffffffu, bwait(bar, parity, abort_flag, p, site));
}

// Teardown wait for the CTA's own copies and MMAs, which always complete.
constexpr unsigned long long kBwdDrainCycles = 2000000000ull;
__device__ __forceinline__ void bdrain(uint64_t* bar, uint32_t parity, const BwdParams& p, int site) {
    const unsigned long long lim = p.wait_limit > kBwdDrainCycles ? p.wait_limit : kBwdDrainCycles;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (static_cast<unsigned long long>(clock64() - t0) > lim) {
            atomicCAS(p.status, 0, site);
            return;
        }
    }
}

// The steps of one CTA: query heads of the group x the query tiles that see
// at least one key of the tile.
struct BwdItem {
    int b, hk, k0;           // batch, key/value head, first key
    int i_lo, n_i;           // query tiles [i_lo, i_lo + n_i)
    int steps;               // group * n_i
    int rot;                 // first query tile offset (spreads the dQ adds)
    // Query head and first query row of step t.  The CTAs of one head start
    // their walk over the query tiles at different tiles, so that their bulk
    // adds into the float32 dQ accumulator do not all hit the same rows.
    __device__ __forceinline__ int head(int t, int group) const { return hk * group + t / n_i; }
    __device__ __forceinline__ int q0(int t, int bm) const {
        int i = t % n_i + rot;
        if (i >= n_i) i -= n_i;
        return (i_lo + i) * bm;
    }
};

template <class Cfg>
__device__ __forceinline__ BwdItem bwd_item(const BwdParams& p) {
    BwdItem w;
    // Head-major order: the CTAs running together share a few heads, so the
    // heads' Q, dO and float32 dQ accumulators stay in L2 while every key
    // tile of the head walks them.
    const int kb = static_cast<int>(blockIdx.x) % p.n_kblocks;
    const int bhk = static_cast<int>(blockIdx.x) / p.n_kblocks;
    w.b = bhk / p.H_kv;
    w.hk = bhk % p.H_kv;
    w.k0 = kb * Cfg::BN;
    const int k1 = min(w.k0 + Cfg::BN, p.N) - 1;
    const int nq = (p.N + Cfg::BM - 1) / Cfg::BM;
    const int lo = p.causal ? w.k0 / Cfg::BM : 0;
    int hi = nq - 1;
    if (p.window > 0) hi = min(hi, (k1 + p.window - 1) / Cfg::BM);
    w.i_lo = lo;
    w.n_i = hi >= lo ? hi - lo + 1 : 0;
    w.steps = w.n_i * p.group;
    // Key tile kb starts at query tile kb * BN / BM of its range: at any
    // moment the CTAs of one head are on different query tiles.
    w.rot = w.n_i > 0 ? static_cast<int>((static_cast<long long>(kb) * (Cfg::BN / Cfg::BM)) % w.n_i) : 0;
    return w;
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                    const BwdParams p) {
    constexpr int D = Cfg::D, BM = Cfg::BM, BN = Cfg::BN, NST = Cfg::NST;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sK = smem + Cfg::OFF_K;
    uint8_t* sV = smem + Cfg::OFF_V;
    uint8_t* sStage = smem + Cfg::OFF_STAGE;
    uint8_t* sDS = smem + Cfg::OFF_DS;
    uint8_t* sDQ = smem + Cfg::OFF_DQ;
    float* sVec = reinterpret_cast<float*>(smem + Cfg::OFF_VEC);
    BwdBarriers* bars = reinterpret_cast<BwdBarriers*>(smem + Cfg::OFF_BAR);
    volatile int* abort_flag = &bars->abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const BwdItem w = bwd_item<Cfg>(p);

    if (threadIdx.x == 0) {
        mbar_init(&bars->kv_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->q_full[s], 1);
            mbar_init(&bars->q_empty[s], 1 + 4 * Cfg::EW_WGS);   // the MMAs' commit + every elementwise warp
            mbar_init(&bars->s_full[s], 1);
            mbar_init(&bars->p_full[s], 128 * Cfg::EW_WGS);
        }
        mbar_init(&bars->dp_full, 1);
        mbar_init(&bars->ds_full, 128 * Cfg::EW_WGS);
        mbar_init(&bars->dq_full, 1);
        mbar_init(&bars->dq_empty, 128);
        mbar_init(&bars->acc_full, 1);
        mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == Cfg::LOAD_WARP && lane == 0) {
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
        tma_prefetch_desc(&tmap_do);
    }
    if (warp == 0) {
        tmem_alloc(&bars->tmem_base, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const int T = w.steps;

    if (warp >= Cfg::LOAD_WARP) {
    if constexpr (Cfg::REG_SPLIT) regs_decrease<Cfg::LM_REGS>();
    if (warp == Cfg::LOAD_WARP) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && T > 0) {
            const uint64_t pol_stream = l2_policy_evict_first();
            const uint64_t pol_keep = l2_policy_evict_last();
            mbar_arrive_expect_tx(&bars->kv_full, 2 * Cfg::KV_TILE);
#pragma unroll
            for (int cb = 0; cb < Cfg::NCB; ++cb) {
                tma_load_4d(sK + cb * (BN * 128), &tmap_k, &bars->kv_full, cb * 64, w.hk, w.k0, w.b, pol_stream);
                tma_load_4d(sV + cb * (BN * 128), &tmap_v, &bars->kv_full, cb * 64, w.hk, w.k0, w.b, pol_stream);
            }
            int t = 0;
            for (; t < T; ++t) {
                const int st = t % NST;
                if (!bwait(&bars->q_empty[st], ((t / NST) & 1) ^ 1, abort_flag, p, BSITE_LOAD_EMPTY)) break;
                const int h = w.head(t, p.group);
                const int q0 = w.q0(t, BM);
                uint8_t* dst = sStage + st * Cfg::STAGE;
                mbar_arrive_expect_tx(&bars->q_full[st], Cfg::STAGE + Cfg::VEC_BYTES);
#pragma unroll
                for (int cb = 0; cb < Cfg::NCB; ++cb) {
                    tma_load_4d(dst + cb * (BM * 128), &tmap_q, &bars->q_full[st], cb * 64, h, q0, w.b, pol_keep);
                    tma_load_4d(dst + Cfg::Q_TILE + cb * (BM * 128), &tmap_do, &bars->q_full[st], cb * 64, h, q0,
                                w.b, pol_keep);
                }
                const size_t row = (static_cast<size_t>(w.b) * p.H + h) * p.N_pad + q0;
                bulk_load(sVec + st * (2 * BM), p.lse2 + row, BM * 4, &bars->q_full[st]);
                bulk_load(sVec + st * (2 * BM) + BM, p.dvec + row, BM * 4, &bars->q_full[st]);
            }
            // Every copy issued lands before the CTA can exit.
            bdrain(&bars->kv_full, 0, p, BSITE_LOAD_DRAIN);
            for (int k = t - NST > 0 ? t - NST : 0; k < t; ++k)
                bdrain(&bars->q_full[k % NST], (k / NST) & 1, p, BSITE_LOAD_DRAIN);
        }
        __syncwarp();
    } else if (warp == Cfg::MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        if (T > 0) {
            const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aDS = smem_u32(sDS);
            const uint64_t k_kmaj = sdesc_sw128(aK, 16, 1024);
            const uint64_t v_kmaj = sdesc_sw128(aV, 16, 1024);
            const uint64_t k_mn = sdesc_sw128(aK, BN * 128, 1024);          // K read MN-major (dQ^T: A; dQ: B)

            constexpr uint32_t id_s = make_idesc_ab(1, 128, BM, 0, 0);      // S^T, dP^T
            constexpr uint32_t id_acc = make_idesc_ab(1, 128, D, 0, 1);     // dV, dK (B MN-major)
            // dS^T buffer of step t: rows = keys, BM queries each (64-query chunks).
            auto ds_addr = [&](int t) { return aDS + (t & 1) * Cfg::DS_BYTES; };
            // dQ^T = K^T dS^T (M = d) or dQ = dS K (M = BM); both operands MN-major.
            constexpr uint32_t id_dq = Cfg::DQ_T ? make_idesc_ab(1, D, BM, 1, 1) : make_idesc_ab(1, BM, D, 1, 1);
            bool ok = bwait_warp(&bars->kv_full, 0, abort_flag, p, BSITE_MMA_KV);

            // S^T = K Q^T or dP^T = V dO^T into `d_col`: d / 16 MMAs, both operands K-major.
            auto issue_kq = [&](uint32_t d_col, uint64_t a_desc, uint32_t b_addr) {
                const uint64_t b_desc = sdesc_sw128(b_addr, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int byte_k = kk * 32;
                    const uint32_t a_off = (byte_k / 128) * (BN * 128) + (byte_k % 128);
                    const uint32_t b_off = (byte_k / 128) * (BM * 128) + (byte_k % 128);
                    mma_f16_ss(tmem + d_col, a_desc + (a_off >> 4), b_desc + (b_off >> 4), id_s, kk > 0 ? 1u : 0u);
                }
            };
            // acc (+)= X^T Y with X^T (bf16 pairs) in tensor memory at x_col and
            // Y (BM query rows x d) in shared memory, read MN-major.
            // P^T of query columns [EC g, EC g + EC) sits at columns
            // [EC g, EC g + EC / 2) of its S^T buffer (written by warpgroup g).
            auto issue_acc = [&](uint32_t d_col, uint32_t x_col, uint32_t y_addr, bool accumulate) {
                const uint64_t y_desc = sdesc_sw128(y_addr, BM * 128, 1024);
#pragma unroll
                for (int kk = 0; kk < BM / 16; ++kk) {
                    constexpr int per_wg = Cfg::EW_COLS / 16;
                    const uint32_t a_col = x_col + (kk / per_wg) * Cfg::EW_COLS + (kk % per_wg) * 8;
                    mma_f16_ts(tmem + d_col, tmem + a_col, y_desc + ((kk * 16 * 128) >> 4), id_acc,
                               (accumulate || kk > 0) ? 1u : 0u);
                }
            };
            auto stage_addr = [&](int t) { return smem_u32(sStage + (t % NST) * Cfg::STAGE); };

            if (ok) ok = bwait_warp(&bars->q_full[0], 0, abort_flag, p, BSITE_MMA_Q);
            if (ok) {
                tc_fence_after();
                if (elect_one()) {
                    issue_kq(Cfg::S_COL, k_kmaj, stage_addr(0));
                    mma_commit(&bars->s_full[0]);   // buffer 0 for step 0 either way
                    issue_kq(Cfg::DP_COL, v_kmaj, stage_addr(0) + Cfg::Q_TILE);
                    mma_commit(&bars->dp_full);
                }
                __syncwarp();
            }
            constexpr int SB = Cfg::S_BUFS;
            for (int t = 0; t < T && ok; ++t) {
                const uint32_t sa = stage_addr(t);
                const uint32_t s_col = Cfg::S_COL + (t % SB) * BM;
                // dV += P^T dO
                if (!bwait_warp(&bars->p_full[t % SB], (t / SB) & 1, abort_flag, p, BSITE_MMA_P)) { ok = false; break; }
                tc_fence_after();
                if (elect_one()) issue_acc(Cfg::DV_COL, s_col, sa + Cfg::Q_TILE, t > 0);
                __syncwarp();
                // S^T of the next step (into the other buffer when there are two;
                // with one, after dV has been issued, which the pipe runs first)
                if (t + 1 < T) {
                    if (!bwait_warp(&bars->q_full[(t + 1) % NST], ((t + 1) / NST) & 1, abort_flag, p, BSITE_MMA_Q)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (elect_one()) {
                        issue_kq(Cfg::S_COL + ((t + 1) % SB) * BM, k_kmaj, stage_addr(t + 1));
                        mma_commit(&bars->s_full[(t + 1) % SB]);
                    }
                    __syncwarp();
                }
                // dS(t) is in shared memory and dP^T(t) has been read: dP^T of
                // the next step first, then dK += dS^T Q and dQ^T = K^T dS^T.
                if (!bwait_warp(&bars->ds_full, t & 1, abort_flag, p, BSITE_MMA_DS)) { ok = false; break; }
                tc_fence_after();
                if (elect_one()) {
                    if (t + 1 < T) {
                        issue_kq(Cfg::DP_COL, v_kmaj, stage_addr(t + 1) + Cfg::Q_TILE);
                        mma_commit(&bars->dp_full);
                    }
                    const uint64_t ds_k = sdesc_sw128(ds_addr(t), 16, 1024);
                    const uint64_t q_mn = sdesc_sw128(sa, BM * 128, 1024);
#pragma unroll
                    for (int kk = 0; kk < BM / 16; ++kk) {
                        const uint32_t a_off = ((kk * 32) / 128) * Cfg::DS_CHUNK + (kk * 32) % 128;
                        mma_f16_ss(tmem + Cfg::DK_COL, ds_k + (a_off >> 4), q_mn + ((kk * 16 * 128) >> 4), id_acc,
                                   (t > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                __syncwarp();
                if (!bwait_warp(&bars->dq_empty, (t & 1) ^ 1, abort_flag, p, BSITE_MMA_DQ)) { ok = false; break; }
                tc_fence_after();
                if (elect_one()) {
                    const uint64_t ds_mn = sdesc_sw128(ds_addr(t), Cfg::DS_CHUNK, 1024);
                    const uint64_t a_dq = Cfg::DQ_T ? k_mn : ds_mn, b_dq = Cfg::DQ_T ? ds_mn : k_mn;
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_f16_ss(tmem + Cfg::DQ_COL, a_dq + ((kk * 16 * 128) >> 4), b_dq + ((kk * 16 * 128) >> 4),
                                   id_dq, kk > 0 ? 1u : 0u);
                    mma_commit(&bars->dq_full);
                    // Q_t and dO_t are no longer read by any MMA.
                    mma_commit(&bars->q_empty[t % NST]);
                    if (t + 1 == T) mma_commit(&bars->acc_full);
                }
                __syncwarp();
            }
            // Every MMA issued has finished before teardown.
            if (elect_one()) {
                mma_commit(&bars->drain);
                bdrain(&bars->drain, 0, p, BSITE_MMA_DRAIN);
            }
            __syncwarp();
        }
    }
    } else if (warp < Cfg::DQ_WARP0) {
        if constexpr (Cfg::REG_SPLIT) regs_increase<Cfg::EW_REGS>();
        // ------------------------------------------------------------ elementwise: P, dS
        constexpr int EC = Cfg::EW_COLS;                 // query columns of this warpgroup
        const int g = warp >> 2;                         // warpgroup: columns [g EC, g EC + EC)
        const int quad = warp & 3;
        const int r = quad * 32 + lane;                  // key row of the tile
        const int key = w.k0 + r;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        bool ok = true;
        constexpr int SB = Cfg::S_BUFS;
        for (int t = 0; t < T && ok; ++t) {
            const int st = t % NST;
            const int q0 = w.q0(t, BM) + g * EC;
            const uint32_t s_tm = tmem + lane_off + Cfg::S_COL + (t % SB) * BM + g * EC;
            const uint32_t dp_tm = tmem + lane_off + Cfg::DP_COL + g * EC;
            if (!bwait_warp(&bars->q_full[st], (t / NST) & 1, abort_flag, p, BSITE_EW_Q)) { ok = false; break; }
            if (!bwait_warp(&bars->s_full[t % SB], (t / SB) & 1, abort_flag, p, BSITE_EW_S)) { ok = false; break; }
            tc_fence_after();
            const float* lse2 = sVec + st * (2 * BM) + g * EC;
            const float* dvec = sVec + st * (2 * BM) + BM + g * EC;
            // Visible queries of this key: [qlo, qhi].
            const int qlo = p.causal ? key : 0;
            const int qhi = p.window > 0 ? key + p.window - 1 : 0x7fffffff;
            const bool key_ok = key < p.N;
            const bool full = key_ok && q0 >= qlo && q0 + EC - 1 <= qhi;
            float pr[EC];
            // 32 columns at a time: read S^T, then write P^T (bf16 pairs) over
            // the first half of this warpgroup's own S^T columns -- the part
            // already read -- so the two warpgroups never overwrite each
            // other's scores.
#pragma unroll
            for (int c = 0; c < EC / 32; ++c) {
                uint32_t sr[32];
                tmem_ld32(s_tm + c * 32, sr);
                tmem_wait_ld();
                reg_fence32(sr);
                uint32_t pk[16];
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                    const int qi = c * 32 + x;
                    float v = ex2_approx(fmaf(__uint_as_float(sr[x]), p.scale_log2, -lse2[qi]));
                    if (!full) {
                        const int q = q0 + qi;
                        if (!key_ok || q < qlo || q > qhi) v = 0.0f;
                    }
                    pr[qi] = v;
                }
#pragma unroll
                for (int x = 0; x < 16; ++x) pk[x] = pack_bf16x2(pr[c * 32 + 2 * x], pr[c * 32 + 2 * x + 1]);
                tmem_st16(s_tm + c * 16, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bars->p_full[t % SB]);

            if (!bwait_warp(&bars->dp_full, t & 1, abort_flag, p, BSITE_EW_DP)) { ok = false; break; }
            tc_fence_after();
            // dS^T(t) goes to buffer t & 1; the MMAs of step t - 2 that read
            // it were issued before dP^T(t), whose completion this thread has
            // just observed.
            uint8_t* ds_buf = sDS + (t & 1) * Cfg::DS_BYTES;
#pragma unroll
            for (int c = 0; c < EC / 32; ++c) {
                uint32_t dr[32];
                tmem_ld32(dp_tm + c * 32, dr);
                tmem_wait_ld();
                reg_fence32(dr);
                uint32_t pk[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const int qi = c * 32 + 2 * x;
                    const float d0 = pr[qi] * (__uint_as_float(dr[2 * x]) - dvec[qi]);
                    const float d1 = pr[qi + 1] * (__uint_as_float(dr[2 * x + 1]) - dvec[qi + 1]);
                    pk[x] = pack_bf16x2(d0, d1);
                }
                // dS^T row of this key into shared memory: 16-byte piece j of
                // the row sits in 64-query chunk j / 8 at position
                // (j % 8) ^ (key % 8) (128-byte swizzle).
#pragma unroll
                for (int y = 0; y < 4; ++y) {
                    const int piece = (g * EC + c * 32) / 8 + y;
                    uint8_t* dst = ds_buf + (piece / 8) * Cfg::DS_CHUNK + r * 128 + (((piece % 8) ^ (r & 7)) * 16);
                    *reinterpret_cast<uint4*>(dst) = make_uint4(pk[4 * y], pk[4 * y + 1], pk[4 * y + 2], pk[4 * y + 3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bars->ds_full);
            // This warp no longer reads the stage's LSE / D.
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->q_empty[st]);
        }
        // dV epilogue (warpgroup 0): thread = key row.
        if (g == 0) {
            if (ok && T > 0) ok = bwait_warp(&bars->acc_full, 0, abort_flag, p, BSITE_EW_ACC);
            if (ok || T == 0) {
                tc_fence_after();
                const bool store = key < p.N;
                __nv_bfloat16* row =
                    reinterpret_cast<__nv_bfloat16*>(p.dv) + ((static_cast<size_t>(w.b) * p.N + key) * p.H_kv + w.hk) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t a[32];
                    if (T > 0) {
                        tmem_ld32(tmem + lane_off + Cfg::DV_COL + c * 32, a);
                        tmem_wait_ld();
                        reg_fence32(a);
                    } else {
#pragma unroll
                        for (int x = 0; x < 32; ++x) a[x] = 0u;
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) pk[x] = pack_bf16x2(__uint_as_float(a[2 * x]), __uint_as_float(a[2 * x + 1]));
                    if (store) {
                        uint4* dst = reinterpret_cast<uint4*>(row + c * 32);
#pragma unroll
                        for (int x = 0; x < 4; ++x) dst[x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
                    }
                }
            }
        }
    } else {
        if constexpr (Cfg::REG_SPLIT) regs_decrease<Cfg::DQ_REGS>();
        // ------------------------------------------------------------ dQ: tensor memory -> bulk add
        const int quad = warp & 3;
        const int r = quad * 32 + lane;                  // dimension (dQ^T) or query (dQ); key row (dK)
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const bool leader = threadIdx.x == Cfg::DQ_WARP0 * 32;
        bool ok = true;
        for (int t = 0; t < T && ok; ++t) {
            const int h = w.head(t, p.group);
            const int q0 = w.q0(t, BM);
            if constexpr (Cfg::DQ_T) {
                // dQ^T: thread = head dimension r, BM query values.
                const bool got = bwait_warp(&bars->dq_full, t & 1, abort_flag, p, BSITE_DQ_FULL);
                // The staging buffer of this step was last read by the bulk add of
                // step t - 2; at most one (step t - 1's) may still be reading.
                if (leader) bulk_wait_group_read<1>();
                // One decision for the four warps (a warp that gave up must not
                // leave the others waiting at the barriers below); the barrier
                // also tells everyone that the staging buffer is free.
                if (!named_barrier_and(1, 128, got)) { ok = false; break; }
                tc_fence_after();
                uint32_t a[BM];
#pragma unroll
                for (int c = 0; c < BM / 32; ++c) tmem_ld32(tmem + lane_off + Cfg::DQ_COL + c * 32, a + c * 32);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < BM / 32; ++c) reg_fence32(a + c * 32);
                tc_fence_before();
                mbar_arrive(&bars->dq_empty);
                float* stage = reinterpret_cast<float*>(sDQ + (t & 1) * Cfg::DQ_STAGE);
#pragma unroll
                for (int x = 0; x < BM; ++x) stage[x * D + r] = __uint_as_float(a[x]);
                fence_proxy_async_smem();
                named_barrier(1, 128);
                if (leader) {
                    float* dst = p.dq_acc + ((static_cast<size_t>(w.b) * p.H + h) * p.N_pad + q0) * D;
                    bulk_reduce_add_f32(dst, stage, Cfg::DQ_STAGE);
                    bulk_commit_group();
                }
            } else {
                // dQ: thread = query row r of the step, d values.  Each thread
                // stages its own row (padded rows: the warp's 16-byte stores
                // spread over the banks) and adds it with its own bulk add, so
                // the four warps need no barrier between them.
                if (!bwait_warp(&bars->dq_full, t & 1, abort_flag, p, BSITE_DQ_FULL)) { ok = false; break; }
                tc_fence_after();
                uint32_t a[D];
#pragma unroll
                for (int c = 0; c < D / 32; ++c) tmem_ld32(tmem + lane_off + Cfg::DQ_COL + c * 32, a + c * 32);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) reg_fence32(a + c * 32);
                tc_fence_before();
                mbar_arrive(&bars->dq_empty);
                // This thread's previous bulk add has finished reading its row.
                bulk_wait_group_read<0>();
                uint8_t* row = sDQ + r * Cfg::DQ_ROW;
#pragma unroll
                for (int x = 0; x < D / 4; ++x)
                    *reinterpret_cast<uint4*>(row + x * 16) = make_uint4(a[4 * x], a[4 * x + 1], a[4 * x + 2], a[4 * x + 3]);
                fence_proxy_async_smem();
                if (q0 + r < p.N_pad) {
                    float* dst = p.dq_acc + ((static_cast<size_t>(w.b) * p.H + h) * p.N_pad + q0 + r) * D;
                    bulk_reduce_add_f32(dst, row, D * 4);
                    bulk_commit_group();
                }
            }
        }
        if (Cfg::DQ_T ? leader : true) bulk_wait_group_all();
        // dK epilogue: thread = key row, scaled by the softmax scale.
        if (ok && T > 0) ok = bwait_warp(&bars->acc_full, 0, abort_flag, p, BSITE_DQ_ACC);
        if (ok || T == 0) {
            tc_fence_after();
            const int key = w.k0 + r;
            const bool store = key < p.N;
            __nv_bfloat16* row =
                reinterpret_cast<__nv_bfloat16*>(p.dk) + ((static_cast<size_t>(w.b) * p.N + key) * p.H_kv + w.hk) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t a[32];
                if (T > 0) {
                    tmem_ld32(tmem + lane_off + Cfg::DK_COL + c * 32, a);
                    tmem_wait_ld();
                    reg_fence32(a);
                } else {
#pragma unroll
                    for (int x = 0; x < 32; ++x) a[x] = 0u;
                }
                uint32_t pk[16];
#pragma unroll
                for (int x = 0; x < 16; ++x)
                    pk[x] = pack_bf16x2(__uint_as_float(a[2 * x]) * p.scale, __uint_as_float(a[2 * x + 1]) * p.scale);
                if (store) {
                    uint4* dst = reinterpret_cast<uint4*>(row + c * 32);
#pragma unroll
                    for (int x = 0; x < 4; ++x) dst[x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
                }
            }
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

}  // namespace attn
