// Fused exact-attention forward for sm_103a (bf16 and FP8 e4m3 inputs).
//
// Method (FlashAttention-3 deep-reading report, "第三层" intro, §3.1, §3.2,
// §3.3; "Efficient Attention & FlashAttention", "数学机理"): K and V are
// streamed tile by tile past a resident tile of queries; every query row keeps
// a running maximum m and a running sum l of its exponentiated scores; the
// output accumulator is rescaled whenever m grows and divided by l once at
// the end.  The N x N score matrix only ever exists one 128 x BN tile at a
// time, in tensor memory.
//
// GB300 mapping (one CTA per SM, warp-specialised):
//   warps [0, 4*NQ)   softmax warpgroups; warpgroup t owns query tile t
//                     (128 rows, one thread per row, TMEM lanes = rows)
//   warp  4*NQ        TMA producer: Q tiles once, then K_j, V_j into an
//                     NSTAGE-deep shared-memory ring (full/empty mbarriers)
//   warp  4*NQ+1      MMA issuer: tcgen05.mma S_t = Q_t K_j^T (both operands
//                     in shared memory) and O_t += P_t V_j (P from tensor
//                     memory, V from shared memory), completion signalled
//                     with tcgen05.commit
// For d >= 128, O leaves through shared memory: each softmax warp owns a
// 4 KB slot (its 32 rows x one 128-byte column box, 128-byte swizzled) and
// hands every box to a TMA store, so the epilogue costs a few shared-memory
// wavefronts per box instead of one scattered global store per row and 16
// bytes.  At d = 64 (one box per row) the direct row stores measured faster.
// Tensor memory (512 columns x 128 lanes of fp32):
//   S_t at columns [128 t, 128 t + BN); P_t (bf16 pairs or e4m3 quads)
//   overwrites the first columns of S_t; O_t at columns [256 + D t, ...).
// The two query tiles alternate on the tensor pipe: while warpgroup 0 runs
// the softmax of S_0(j), the pipe computes O_1 += P_1 V_{j-1} and
// S_1(j) = Q_1 K_j^T (the report's §3.1 ping-pong of softmax against the
// other tile's GEMMs, with the GEMM of one iteration overlapping the softmax
// of the next as in §3.2).
//
// Every barrier wait is bounded: a role that gives up records a site code in
// the status word, raises a shared abort flag and leaves its loop, so the CTA
// always reaches its teardown (TMEM free) instead of hanging.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>
#include <type_traits>

#include "sm103_bulk.cuh"
#include "sm103_ptx.cuh"

namespace attn {

struct FwdParams {
    void* o;                 // bf16 (B, N, H, D)
    float* lse;              // fp32 (B, H, N)
    const float* q_scale;    // FP8 only: (B, H, nblk)
    const float* k_scale;
    const float* v_scale;
    int B, H, N;
    int group;               // query heads per key/value head (1 = multi-head)
    int causal, window;
    float scale_log2;        // softmax scale * log2(e)
    int n_mblocks;           // ceil(N / (NQ * 128))
    const uint8_t* block_mask;   // block-sparse only: (B, H, n_tb, n_tb), nonzero = visible
    int n_tb;                    // ceil(N / 128): 128 x 128 mask blocks per side
    unsigned long long wait_limit;
    int* status;             // device status word (first failing site)
};

// Status site codes: role * 16 + barrier.
enum : int {
    SITE_LOAD_EMPTY = 0x11,
    SITE_LOAD_DRAIN = 0x12,
    SITE_MMA_Q = 0x21,
    SITE_MMA_FULL = 0x22,
    SITE_MMA_P = 0x23,
    SITE_MMA_DRAIN = 0x24,
    SITE_SOFTMAX_S = 0x31,
    SITE_SOFTMAX_O = 0x32,
    SITE_TURN = 0x41,
};

template <int D_, int BN_, int NQ_, bool FP8_, bool SPARSE_ = false>
struct FwdCfg {
    static constexpr bool SPARSE = SPARSE_;               // block-sparse key mask
    static constexpr int D = D_;
    static constexpr int BN = BN_;
    static constexpr int NQ = NQ_;
    static constexpr bool FP8 = FP8_;
    static constexpr int BM = 128;                       // query rows per tile
    static constexpr int ES = FP8 ? 1 : 2;               // bytes per element
    static constexpr int ROW_BYTES = D * ES;
    // Swizzle span: 128-byte column boxes, or one 64-byte box when a row is
    // 64 bytes (e4m3, d = 64).  Tiles are [box][rows][SW bytes].
    static constexpr int SW = ROW_BYTES >= 128 ? 128 : 64;
    static constexpr int NCB = ROW_BYTES / SW;           // column boxes per row
    static constexpr int BOX_ELEMS = SW / ES;
    static constexpr int Q_TILE_BYTES = BM * ROW_BYTES;
    static constexpr int KV_TILE_BYTES = BN * ROW_BYTES;
    // A ring stage holds what key-tile step u consumes: K_u (for S(u)) and
    // V_{u-1} (for P(u-1) V), under one barrier.
    static constexpr int STAGE_BYTES = 2 * KV_TILE_BYTES;
    static constexpr int RING_BUDGET = 196 * 1024 - NQ * Q_TILE_BYTES;
    static constexpr int NSTAGE_RAW = RING_BUDGET / STAGE_BYTES;
    static constexpr int NSTAGE = NSTAGE_RAW > 8 ? 8 : NSTAGE_RAW;
    static constexpr int MMA_K = FP8 ? 32 : 16;          // K per MMA instruction
    static constexpr int P_COLS = BN * ES / 4;           // TMEM columns of one P row
    static constexpr int S_COL = 128;                    // column stride of S_t
    static constexpr int O_COL0 = 256;
    static constexpr int TMEM_COLS = 512;
    static constexpr int NUM_SOFTMAX_THREADS = NQ * 128;
    static constexpr int LOAD_WARP = NQ * 4;
    static constexpr int MMA_WARP = NQ * 4 + 1;   // MMA warps: MMA_WARP .. MMA_WARP + MMA_WARPS - 1
    // Issuer warps: one per query tile where the tile's MMAs are long enough
    // (bf16, d = 128) for the hand-off latency to dominate; one warp for both
    // tiles where the softmax is the longer phase (FP8, d = 64) or NQ = 1.
    static constexpr int MMA_WARPS = (!FP8 && D == 128 && NQ == 2) ? 2 : 1;
    static constexpr int THREADS = NQ * 128 + 128;
    static constexpr int BAR_BYTES = 256;
    // Output staging (O_VIA_TMA): one slot of 32 rows x 128 bytes per
    // softmax warp.
    static constexpr bool O_VIA_TMA = D >= 128;
    static constexpr int EPI_SLOT_BYTES = 32 * 128;
    static constexpr int EPI_BYTES = O_VIA_TMA ? NQ * 4 * EPI_SLOT_BYTES : 0;
    // The reference maximum of a row moves only when the row maximum exceeds
    // it by more than this (log2 units), so P <= 2^RESCALE_LOG2.  FP8 scales P
    // by P8_SCALE = 16 before the e4m3 cast: P * P8_SCALE <= 2^4.8 * 16 ~ 445.7
    // < 448, the largest e4m3 value (and the V factor folded in is <= 1).
    static constexpr float RESCALE_LOG2 = FP8 ? 4.8f : 8.0f;
    static constexpr float P8_SCALE = FP8 ? 16.0f : 1.0f;
    // FP8: when the reference moves, it is set this far (log2 units) above
    // the new row maximum, so that the next moves need a larger jump (the
    // outlier workload's maxima grow in jumps); the tile's P are then <= 1/8.
    static constexpr float RESCALE_HEADROOM = FP8 ? 3.0f : 0.0f;
    // Register split: the launch gives every thread LAUNCH_REGS; the load /
    // MMA warpgroup drops to LOW_REGS and the softmax warpgroups rise to
    // HIGH_REGS.  The sum stays within the launch allocation.
    static constexpr int LAUNCH_REGS = (65536 / THREADS) / 8 * 8 > 255 ? 248 : (65536 / THREADS) / 8 * 8;
    static constexpr int LOW_REGS = FP8 ? 72 : 104;
    static constexpr int HIGH_REGS_RAW = ((LAUNCH_REGS * THREADS - LOW_REGS * 128) / (NQ * 128)) / 8 * 8;
    static constexpr int HIGH_REGS = HIGH_REGS_RAW > 248 ? 248 : HIGH_REGS_RAW;
    static_assert(HIGH_REGS * NQ * 128 + LOW_REGS * 128 <= LAUNCH_REGS * THREADS, "register split");
    static constexpr int SMEM_BYTES = 1024 + NQ * Q_TILE_BYTES + NSTAGE * STAGE_BYTES + EPI_BYTES + BAR_BYTES;

    static_assert(D == 64 || D == 128 || D == 256, "head_dim");
    static_assert(BN == 64 || BN == 128, "key tile");
    static_assert(NCB >= 1 && ROW_BYTES % SW == 0, "rows must be whole swizzle boxes");
    static_assert(NQ * 128 + 0 <= 256 && O_COL0 + NQ * D <= TMEM_COLS, "tensor memory budget");
    static_assert(NSTAGE >= 2, "ring depth");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

struct SharedBarriers {
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_full[2];
    uint64_t drain[2];
    uint64_t ring_full[8];
    uint64_t ring_empty[8];
    uint32_t tmem_base;
    int abort_flag;
    int issued_blocks;    // MMA blocks issued so far (ping-pong turn counter)
};

// Bounded wait on an mbarrier phase.  Returns false when the shared abort
// flag is raised or the cycle budget runs out (then it raises the flag and
// records `site`).
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                           const FwdParams& p, int site) {
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

// wait_phase for a converged warp: every lane polls; the result is the same
// in every lane (a lane that gave up makes the whole warp give up).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          const FwdParams& p, int site) {
    const bool w = wait_phase(bar, parity, abort_flag, p, site);
    return __all_sync(0xffffffffu, w);
}

// Teardown wait for the CTA's own asynchronous work (TMA copies it issued,
// MMAs it committed).  That work always completes, so this wait ignores the
// abort flag and uses at least kDrainCycles even when the per-wait limit has
// been made small, so that no CTA exits with copies or MMAs in flight.
constexpr unsigned long long kDrainCycles = 2000000000ull;
__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity, const FwdParams& p, int site) {
    const unsigned long long lim = p.wait_limit > kDrainCycles ? p.wait_limit : kDrainCycles;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (static_cast<unsigned long long>(clock64() - t0) > lim) {
            atomicCAS(p.status, 0, site);
            return false;
        }
    }
    return true;
}

// FP8: the largest V block scale of one (batch, key/value head), the
// normaliser of the V factors folded into P (P8 = e4m3(P * P8_SCALE *
// v_scale_j / vmax)).  Every lane of the warp loads every 32nd block scale
// and the warp reduces them, so each warp gets the same value without any
// cross-warp synchronisation.  1 when every scale is 0.
__device__ __forceinline__ float fp8_vmax(const float* vs, int nblk) {
    float v = 0.0f;
    for (int x = static_cast<int>(lane_id()); x < nblk; x += 32) v = fmaxf(v, __ldg(vs + x));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v > 0.0f ? v : 1.0f;
}

// FP8: the factors of one key tile's softmax step, from the K and V block
// scales of the 128-key block `sb`: mult takes the raw e4m3 scores to log2
// units (softmax scale * log2 e * q_scale * k_scale), lg = log2(pv_mult) is
// added to the exponent so that exp2 yields P * pv_mult directly (the V
// block's factor, pv_mult = P8_SCALE * v_scale / vmax, folded into P), and
// inv = 2^-lg turns the tile's sum back into a sum of P (the inverse of the
// factor actually applied, so P's weights and l stay consistent).  inv_vmax
// is 1 / vmax, taken once per item: no division per key tile.  The softmax
// loads these one step ahead, while it waits for the next S, so that no
// global load or logarithm lies between an S becoming visible and its P
// being handed over.
template <class Cfg>
__device__ __forceinline__ void fp8_tile_scales(const FwdParams& p, size_t sb, float q_mult, float inv_vmax,
                                                float& mult, float& lg, float& inv) {
    mult = q_mult * __ldg(p.k_scale + sb);
    const float pv_mult = Cfg::P8_SCALE * (__ldg(p.v_scale + sb) * inv_vmax);
    lg = __log2f(pv_mult);
    inv = ex2_approx(-lg);
}

// Makes three values available at this point of the program (the compiler
// may not sink their computation below it, e.g. past a barrier wait).
__device__ __forceinline__ void pin3(float& a, float& b, float& c) { asm volatile("" : "+f"(a), "+f"(b), "+f"(c)); }

template <class Cfg>
__device__ __forceinline__ void tile_range(const FwdParams& p, int qs, int& lo, int& hi) {
    const int qe = min(qs + Cfg::BM, p.N) - 1;
    lo = p.window > 0 ? max(0, qs - p.window + 1) / Cfg::BN : 0;
    hi = p.causal ? qe / Cfg::BN : (p.N - 1) / Cfg::BN;
}

// Work items are (query block of NQ*128 rows, batch*head).  Causal items
// are numbered heaviest query block first, non-causal items head by head so
// that the CTAs running together share K and V in L2.  CTA c takes, in round
// m, item m*G + c when m is even and m*G + G-1-c when m is odd (G = grid):
// the zigzag gives the CTA that got the lightest item of one round the
// heaviest of the next, which balances causal work without any scheduler
// state in memory.
__device__ __forceinline__ int round_item(int m) {
    const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    return m * G + ((m & 1) ? (G - 1 - c) : c);
}

// A causal launch's work order, computed on the host (causal_item_order): the n
// mod G lightest items (query block ascending, then head) form the last,
// partial round; the others, taken head by head (query block descending
// within a head), are cut into rounds of G, each numbered heaviest query
// block first, then by head.  The zigzag still balances (every round is
// numbered heaviest first), and a round touches the K and V of about
// G / n_mblocks heads instead of all of them.  e[item] = query block |
// (batch*head) << 16.  n = 0: the closed-form order of item_coords.  It rides
// in the launch's parameters (no memory shared between launches).
constexpr int kOrderMax = 2048;
struct ItemOrder {
    int n;
    uint32_t e[kOrderMax];
};
// The parameter of a kernel built without an order table (4 bytes instead of
// 8 KB: the other launches do not pay for the table).
struct NoOrder {
    int n;
};

__device__ __forceinline__ void item_coords(const FwdParams& p, int item, int& mb, int& bh) {
    const int BH = p.B * p.H;
    if (p.causal) {
        mb = p.n_mblocks - 1 - item / BH;
        bh = item % BH;
    } else {
        mb = item % p.n_mblocks;
        bh = item / p.n_mblocks;
    }
}

// The key tiles of an item.  Query tile t sees key tiles [lo[t], hi[t]]
// (causal / window ranges), and with a block-sparse mask only those whose
// 128 x 128 mask block is set; first[t] / last[t] are its first and last
// visible key tile (-1 when it sees none, which makes the tile inactive).
// The roles walk the union of the active tiles' sets in increasing order;
// -1 ends a walk.
template <int NQ>
struct WorkItem {
    int b, h, bh, q0;
    int lo[NQ], hi[NQ];
    int first[NQ], last[NQ];
    bool active[NQ];
    bool in_n[NQ];        // query tile starts inside the sequence
    const uint8_t* mrow[NQ];
    int u_lo, u_hi;       // first and last key tile of the union (-1: none)
};

template <class Cfg>
__device__ __forceinline__ bool key_in_tile(const WorkItem<Cfg::NQ>& w, int t, int u) {
    if (u < w.lo[t] || u > w.hi[t]) return false;
    if constexpr (Cfg::SPARSE) return __ldg(w.mrow[t] + ((u * Cfg::BN) >> 7)) != 0;
    return true;
}

// Next key tile after u in the union of the active tiles' sets, or -1.
template <class Cfg>
__device__ __forceinline__ int next_key(const WorkItem<Cfg::NQ>& w, int u) {
    if constexpr (!Cfg::SPARSE) {
        return u < w.u_hi ? u + 1 : -1;
    } else {
        for (int x = u + 1; x <= w.u_hi; ++x) {
#pragma unroll
            for (int t = 0; t < Cfg::NQ; ++t)
                if (w.active[t] && key_in_tile<Cfg>(w, t, x)) return x;
        }
        return -1;
    }
}

// One query tile's part of an item, for roles that index the tile at run
// time (a register copy instead of a dynamically indexed array).
struct TileKeys {
    int lo, hi, first, last;
    bool active, in_n;
    const uint8_t* mrow;
};

template <class Cfg>
__device__ __forceinline__ TileKeys tile_keys(const WorkItem<Cfg::NQ>& w, int t) {
    TileKeys k{w.lo[0], w.hi[0], w.first[0], w.last[0], w.active[0], w.in_n[0], w.mrow[0]};
#pragma unroll
    for (int x = 1; x < Cfg::NQ; ++x)
        if (t == x) k = TileKeys{w.lo[x], w.hi[x], w.first[x], w.last[x], w.active[x], w.in_n[x], w.mrow[x]};
    return k;
}

// Next key tile after u in the tile's set, or -1.
template <class Cfg>
__device__ __forceinline__ int next_in(const TileKeys& k, int u) {
    if constexpr (!Cfg::SPARSE) {
        return u < k.last ? u + 1 : -1;
    } else {
        for (int x = u + 1; x <= k.last; ++x)
            if (__ldg(k.mrow + ((x * Cfg::BN) >> 7)) != 0) return x;
        return -1;
    }
}

template <class Cfg, class Order = NoOrder>
__device__ __forceinline__ WorkItem<Cfg::NQ> decode_item(const FwdParams& p, int item,
                                                        const Order* order = nullptr) {
    WorkItem<Cfg::NQ> w;
    int mb;
    if constexpr (std::is_same<Order, ItemOrder>::value) {
        const uint32_t e = order->e[item];
        mb = static_cast<int>(e & 0xffffu);
        w.bh = static_cast<int>(e >> 16);
    } else {
        item_coords(p, item, mb, w.bh);
    }
    w.b = w.bh / p.H;
    w.h = w.bh % p.H;
    w.q0 = mb * Cfg::NQ * Cfg::BM;
    w.u_lo = -1;
    w.u_hi = -1;
#pragma unroll
    for (int t = 0; t < Cfg::NQ; ++t) {
        const int qs = w.q0 + t * Cfg::BM;
        w.in_n[t] = qs < p.N;
        tile_range<Cfg>(p, qs, w.lo[t], w.hi[t]);
        w.mrow[t] = nullptr;
        w.first[t] = w.lo[t];
        w.last[t] = w.hi[t];
        if constexpr (Cfg::SPARSE) {
            w.mrow[t] = p.block_mask + (static_cast<size_t>(w.bh) * p.n_tb + min(qs, p.N - 1) / 128) * p.n_tb;
            w.first[t] = -1;
            w.last[t] = -1;
            if (w.in_n[t]) {
                for (int x = w.lo[t]; x <= w.hi[t]; ++x)
                    if (key_in_tile<Cfg>(w, t, x)) { w.first[t] = x; break; }
                for (int x = w.hi[t]; x >= w.lo[t] && w.first[t] >= 0; --x)
                    if (key_in_tile<Cfg>(w, t, x)) { w.last[t] = x; break; }
            }
        }
        w.active[t] = w.in_n[t] && w.first[t] >= 0 && w.first[t] <= w.last[t];
        if (w.active[t]) {
            w.u_lo = w.u_lo < 0 ? w.first[t] : min(w.u_lo, w.first[t]);
            w.u_hi = max(w.u_hi, w.last[t]);
        }
    }
    return w;
}

// Key-tile walk and MMA issue order (the ping-pong of the two query tiles).
// A CTA walks the steps of its items back to back: one step per key tile u
// of an item (walk order), and one final step after its last item.  A step's
// ring stage holds K_u and the V of the previous step's key tile (which may
// belong to the previous item), and its block for tile t (t = 0, 1 in
// order) holds O_t += P_t V of the previous step (when tile t had an S
// there) followed by S_t = Q_t K_u^T (when u is in tile t's set).  So the
// last P V of one item and the first S of the next share a step, like any
// two consecutive key tiles: the next item's first S of a tile never waits
// for the other tile's last softmax of the previous item, and an item costs
// no extra step for its final P V.  Empty blocks are skipped; the issuers
// count the non-empty blocks and, with two issuers, each waits for its
// blocks' turns in that order.
// Bounded wait (whole warp) until `k` MMA blocks have been issued.
__device__ __forceinline__ bool wait_turn(volatile int* issued, int k, volatile int* abort_flag,
                                          const FwdParams& p, int site) {
    bool ok = true;
    if (*issued < k) {
        const long long t0 = clock64();
        while (*issued < k) {
            if (*abort_flag) { ok = false; break; }
            if (static_cast<unsigned long long>(clock64() - t0) > p.wait_limit) {
                *abort_flag = 1;
                atomicCAS(p.status, 0, site);
                ok = false;
                break;
            }
        }
    }
    return __all_sync(0xffffffffu, ok);
}

// S_t = Q_t K^T: D / MMA_K instructions, operands in shared memory (both
// K-major, 128-byte swizzle); each k-step advances the descriptors' start
// address by a constant.
template <class Cfg>
__device__ __forceinline__ void issue_qk(uint32_t s_tmem, uint64_t qdesc, uint64_t kdesc) {
    constexpr uint32_t fmt = Cfg::FP8 ? 0u : 1u;
    constexpr uint32_t idesc = make_idesc(fmt, 128, Cfg::BN, 0);
#pragma unroll
    for (int kk = 0; kk < Cfg::D / Cfg::MMA_K; ++kk) {
        constexpr int step_bytes = Cfg::MMA_K * Cfg::ES;
        const int byte_k = kk * step_bytes;
        constexpr int SW = Cfg::SW;
        const uint32_t a_off = (byte_k / SW) * (Cfg::BM * SW) + (byte_k % SW);
        const uint32_t b_off = (byte_k / SW) * (Cfg::BN * SW) + (byte_k % SW);
        if constexpr (Cfg::FP8)
            mma_f8_ss(s_tmem, qdesc + (a_off >> 4), kdesc + (b_off >> 4), idesc, kk > 0 ? 1u : 0u);
        else
            mma_f16_ss(s_tmem, qdesc + (a_off >> 4), kdesc + (b_off >> 4), idesc, kk > 0 ? 1u : 0u);
    }
}

// O_t (+)= P_t V: BN / MMA_K instructions, P from tensor memory, V from
// shared memory (MN-major, 128-byte swizzle).
template <class Cfg>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint64_t vdesc, bool accumulate) {
    constexpr uint32_t fmt = Cfg::FP8 ? 0u : 1u;
    constexpr uint32_t idesc = make_idesc(fmt, 128, Cfg::D, 1);
    const uint32_t acc0 = accumulate ? 1u : 0u;
#pragma unroll
    for (int kk = 0; kk < Cfg::BN / Cfg::MMA_K; ++kk) {
        const uint64_t off = (static_cast<uint64_t>(kk) * Cfg::MMA_K * Cfg::SW) >> 4;
        if constexpr (Cfg::FP8)
            mma_f8_ts(o_tmem, p_tmem + kk * (Cfg::MMA_K / 4), vdesc + off, idesc, kk > 0 ? 1u : acc0);
        else
            mma_f16_ts(o_tmem, p_tmem + kk * (Cfg::MMA_K / 2), vdesc + off, idesc, kk > 0 ? 1u : acc0);
    }
}

// ORDERED: the causal work order comes from `order` (a causal launch with a
// host-built table); otherwise from item_coords.
template <class Cfg, bool ORDERED = false>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_o,
                    const FwdParams p,
                    const __grid_constant__ typename std::conditional<ORDERED, ItemOrder, NoOrder>::type order) {
    constexpr int D = Cfg::D, BN = Cfg::BN, NQ = Cfg::NQ, BM = Cfg::BM, NSTAGE = Cfg::NSTAGE;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;                                       // NQ x Q tile
    uint8_t* sKV = smem + NQ * Cfg::Q_TILE_BYTES;             // NSTAGE x (K tile, V tile)
    uint8_t* sEpi = sKV + NSTAGE * Cfg::STAGE_BYTES;        // 4*NQ output slots
    SharedBarriers* bars = reinterpret_cast<SharedBarriers*>(sEpi + Cfg::EPI_BYTES);
    volatile int* abort_flag = &bars->abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bars->q_full[t], 1);
            mbar_init(&bars->q_empty[t], 1);
            mbar_init(&bars->s_full[t], 1);
            mbar_init(&bars->p_full[t], 128);
            mbar_init(&bars->o_full[t], 1);
        }
        mbar_init(&bars->drain[0], 1);
        mbar_init(&bars->drain[1], 1);
        for (int s = 0; s < 8; ++s) {
            mbar_init(&bars->ring_full[s], 1);
            mbar_init(&bars->ring_empty[s], Cfg::MMA_WARPS);
        }
        bars->abort_flag = 0;
        bars->issued_blocks = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == Cfg::LOAD_WARP && lane == 0) {
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
        tma_prefetch_desc(&tmap_o);
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

    if (warp >= 4 * NQ) {
    regs_decrease<Cfg::LOW_REGS>();
    if (warp == Cfg::LOAD_WARP) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            uint32_t it = 0;
            uint32_t qn[NQ];
#pragma unroll
            for (int t = 0; t < NQ; ++t) qn[t] = 0;
            int vb = 0, vh = 0, vu = -1;   // V of the previous step (batch, key/value head, key tile)
            // One ring step: K tile ku of (batch kb, key/value head kh) when
            // with_k, and the previous step's V when there is one.
            auto load_step = [&](bool with_k, int kb, int kh, int ku) -> bool {
                const uint32_t stage = it % NSTAGE, round = it / NSTAGE;
                if (!wait_phase(&bars->ring_empty[stage], (round & 1) ^ 1, abort_flag, p, SITE_LOAD_EMPTY))
                    return false;
                const bool with_v = vu >= 0;
                mbar_arrive_expect_tx(&bars->ring_full[stage],
                                      (with_k ? Cfg::KV_TILE_BYTES : 0) + (with_v ? Cfg::KV_TILE_BYTES : 0));
                uint8_t* dst = sKV + stage * Cfg::STAGE_BYTES;
                if (with_k) {
#pragma unroll
                    for (int cb = 0; cb < Cfg::NCB; ++cb)
                        tma_load_4d(dst + cb * (BN * Cfg::SW), &tmap_k, &bars->ring_full[stage], cb * Cfg::BOX_ELEMS,
                                    kh, ku * BN, kb, pol_kv);
                }
                if (with_v) {
#pragma unroll
                    for (int cb = 0; cb < Cfg::NCB; ++cb)
                        tma_load_4d(dst + Cfg::KV_TILE_BYTES + cb * (BN * Cfg::SW), &tmap_v, &bars->ring_full[stage],
                                    cb * Cfg::BOX_ELEMS, vh, vu * BN, vb, pol_kv);
                }
                ++it;
                return true;
            };
            bool ok = true;
            for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < total_items && ok; ++rnd) {
                const int item = round_item(rnd);
                if (item >= total_items) continue;
                const WorkItem<NQ> w = decode_item<Cfg>(p, item, &order);
#pragma unroll
                for (int t = 0; t < NQ; ++t) {
                    if (!w.active[t] || !ok) continue;
                    // The previous item's S MMAs of this tile must be done.
                    if (!wait_phase(&bars->q_empty[t], (qn[t] & 1) ^ 1, abort_flag, p, SITE_LOAD_EMPTY)) {
                        ok = false;
                        continue;
                    }
                    ++qn[t];
                    mbar_arrive_expect_tx(&bars->q_full[t], Cfg::Q_TILE_BYTES);
#pragma unroll
                    for (int cb = 0; cb < Cfg::NCB; ++cb)
                        tma_load_4d(sQ + t * Cfg::Q_TILE_BYTES + cb * (BM * Cfg::SW), &tmap_q, &bars->q_full[t],
                                    cb * Cfg::BOX_ELEMS, w.h, w.q0 + t * BM, w.b, pol_q);
                }
                // The item's steps: K_u, and the V of the previous step.
                const int kh = w.h / p.group;
                for (int u = w.u_lo; ok && u >= 0; u = next_key<Cfg>(w, u)) {
                    ok = load_step(true, w.b, kh, u);
                    vb = w.b;
                    vh = kh;
                    vu = u;
                }
            }
            // Final step: the V of the last key tile.
            if (ok && vu >= 0) ok = load_step(false, 0, 0, 0);
            // Let every copy this warp issued land before the CTA can exit (on
            // the normal path these phases have completed already).
            const uint32_t first = it > NSTAGE ? it - NSTAGE : 0;
            for (uint32_t k = first; k < it; ++k)
                drain_wait(&bars->ring_full[k % NSTAGE], (k / NSTAGE) & 1, p, SITE_LOAD_DRAIN);
#pragma unroll
            for (int t = 0; t < NQ; ++t)
                if (qn[t] > 0) drain_wait(&bars->q_full[t], (qn[t] - 1) & 1, p, SITE_LOAD_DRAIN);
        }
        __syncwarp();
    } else if (warp >= Cfg::MMA_WARP && warp < Cfg::MMA_WARP + Cfg::MMA_WARPS) {
        // ------------------------------------------------------------ MMA issuers
        // Issuer warp w owns the query tiles t = w, w + MMA_WARPS, ...  Issuing
        // one tcgen05.mma takes tens of cycles, so with long MMAs one warp cannot
        // feed two tiles and also answer their P hand-offs in time; with a warp
        // per tile, one waits for its P while the other issues.  The blocks go
        // to the tensor pipe in the ping-pong order either way (a turn counter
        // in shared memory when there are two issuers), so the two softmax
        // warpgroups stay out of phase.  The whole warp runs the loop
        // (descriptors stay warp-uniform); one elected lane issues the MMAs and
        // the commits.  Each issuer releases every ring stage once (ring_empty
        // counts MMA_WARPS), always after waiting for its load, so no issuer can
        // get a ring cycle ahead.
        constexpr int MW = Cfg::MMA_WARPS;
        const int wi = warp - Cfg::MMA_WARP;
        const uint32_t sKV_addr = smem_u32(sKV);
        volatile int* issued = &bars->issued_blocks;
        uint64_t qdesc[NQ];
#pragma unroll
        for (int t = 0; t < NQ; ++t)
            qdesc[t] = sdesc_swz<Cfg::SW>(smem_u32(sQ) + t * Cfg::Q_TILE_BYTES, 16, 8 * Cfg::SW);
        uint32_t it = 0;
        uint32_t pv_count[NQ], qn[NQ];
        // Bit t: tile t's P V of the previous step is due (pend), accumulates
        // into O_t (pend_acc: not the tile's first key tile of its item) and
        // ends the tile's item (pend_last: O_t is final once it is done).
        uint32_t pend = 0, pend_acc = 0, pend_last = 0;
#pragma unroll
        for (int t = 0; t < NQ; ++t) pv_count[t] = qn[t] = 0;
        int turn = 0;        // non-empty blocks (of both issuers) so far
        // One step.  Bit t of s_mask: tile t has S = Q_t K^T here; of
        // first_mask / last_mask: that key tile is the tile's first / last of
        // its item (all 0 for the final step).
        auto mma_step = [&](uint32_t s_mask, uint32_t first_mask, uint32_t last_mask) -> bool {
            const uint32_t stage = it % NSTAGE, round = it / NSTAGE;
            ++it;
            if (!warp_wait(&bars->ring_full[stage], round & 1, abort_flag, p, SITE_MMA_FULL)) return false;
            const uint32_t st_addr = sKV_addr + stage * Cfg::STAGE_BYTES;
            const uint64_t kdesc = sdesc_swz<Cfg::SW>(st_addr, 16, 8 * Cfg::SW);
            const uint64_t vdesc = sdesc_swz<Cfg::SW>(st_addr + Cfg::KV_TILE_BYTES, BN * Cfg::SW, 8 * Cfg::SW);
            bool issued_any = false;
#pragma unroll
            for (int t = 0; t < NQ; ++t) {
                const bool do_pv = (pend >> t) & 1u;
                const bool do_s = (s_mask >> t) & 1u;
                if (!do_pv && !do_s) continue;
                const int k = turn++;
                if (t % MW != wi) continue;
                if (do_pv && !warp_wait(&bars->p_full[t], pv_count[t] & 1, abort_flag, p, SITE_MMA_P)) return false;
                if (MW > 1 && !wait_turn(issued, k, abort_flag, p, SITE_TURN)) return false;
                tc_fence_after();
                if (elect_one()) {
                    if (do_pv) {
                        issue_pv<Cfg>(tmem + Cfg::O_COL0 + t * D, tmem + t * Cfg::S_COL, vdesc, (pend_acc >> t) & 1u);
                        if ((pend_last >> t) & 1u) mma_commit(&bars->o_full[t]);
                    }
                    if (do_s) {
                        issue_qk<Cfg>(tmem + t * Cfg::S_COL, qdesc[t], kdesc);
                        mma_commit(&bars->s_full[t]);
                        // Q_t is free for the next item once its last S MMA is done.
                        if ((last_mask >> t) & 1u) mma_commit(&bars->q_empty[t]);
                    }
                    if (MW > 1) {
                        __threadfence_block();
                        *issued = k + 1;
                    }
                }
                __syncwarp();
                issued_any = true;
                if (do_pv) ++pv_count[t];
            }
            pend = s_mask;
            pend_acc = s_mask & ~first_mask;
            pend_last = s_mask & last_mask;
            // This issuer is done with the stage once its MMAs of the step are.
            if (elect_one()) {
                if (issued_any) mma_commit(&bars->ring_empty[stage]);
                else mbar_arrive(&bars->ring_empty[stage]);
            }
            __syncwarp();
            return true;
        };
        bool ok = true;
        bool any_step = false;
        for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < total_items && ok; ++rnd) {
            const int item = round_item(rnd);
            if (item >= total_items) continue;
            const WorkItem<NQ> w = decode_item<Cfg>(p, item, &order);
#pragma unroll
            for (int t = 0; t < NQ; ++t) {
                if (t % MW == wi && w.active[t] && ok) {
                    ok = warp_wait(&bars->q_full[t], qn[t] & 1, abort_flag, p, SITE_MMA_Q);
                    ++qn[t];
                }
            }
            for (int u = w.u_lo; ok && u >= 0; u = next_key<Cfg>(w, u)) {
                uint32_t s_mask = 0, first_mask = 0, last_mask = 0;
#pragma unroll
                for (int t = 0; t < NQ; ++t) {
                    if (w.active[t] && key_in_tile<Cfg>(w, t, u)) s_mask |= 1u << t;
                    if (u == w.first[t]) first_mask |= 1u << t;
                    if (u == w.last[t]) last_mask |= 1u << t;
                }
                ok = mma_step(s_mask, first_mask, last_mask);
                any_step = true;
            }
        }
        // Final step: the last P V of each tile.
        if (ok && any_step) ok = mma_step(0u, 0u, 0u);
        // Every MMA this warp issued has finished before teardown.
        if (elect_one()) {
            mma_commit(&bars->drain[wi]);
            drain_wait(&bars->drain[wi], 0, p, SITE_MMA_DRAIN);
        }
        __syncwarp();
    }
    } else {
        regs_increase<Cfg::HIGH_REGS>();
        // ------------------------------------------------------------ softmax
        const int t = warp >> 2;
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t s_tmem = tmem + lane_off + t * Cfg::S_COL;
        const uint32_t o_tmem = tmem + lane_off + Cfg::O_COL0 + t * D;
        const int nblk = (p.N + 127) / 128;
        uint32_t count = 0;    // S tiles consumed (s_full phases)
        uint32_t qn = 0;       // items in which this tile was active (o_full phases)
        bool ok = true;
        for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < total_items && ok; ++rnd) {
            const int item = round_item(rnd);
            if (item >= total_items) continue;
            const WorkItem<NQ> w = decode_item<Cfg>(p, item, &order);
            const TileKeys tk = tile_keys<Cfg>(w, t);
            const int bh = w.bh, b = w.b, h = w.h;
            const int qs = w.q0 + t * BM;
            if (!tk.in_n) continue;                          // tile t beyond the sequence
            const int i = qs + r;                                  // query row
            if (!tk.active) {
                // Block-sparse mask: this query tile sees no key.
                if (i < p.N) {
                    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) +
                                                          ((static_cast<size_t>(b) * p.N + i) * p.H + h) * D);
#pragma unroll
                    for (int x = 0; x < D / 8; ++x) dst[x] = make_uint4(0u, 0u, 0u, 0u);
                    p.lse[static_cast<size_t>(bh) * p.N + i] = -INFINITY;
                }
                continue;
            }
            // Visible keys of row i: [klo, khi].
            const int klo = p.window > 0 ? i - p.window + 1 : 0;
            const int khi = p.causal ? min(i, p.N - 1) : p.N - 1;
            float vmax = 1.0f, ivmax = 1.0f;
            float q_mult = p.scale_log2;
            // Key/value head of this query head (grouped-query attention).
            const int bh_kv = b * (p.H / p.group) + h / p.group;
            const size_t sb0 = static_cast<size_t>(bh_kv) * nblk;
            if constexpr (Cfg::FP8) {
                vmax = fp8_vmax(p.v_scale + sb0, nblk);
                ivmax = 1.0f / vmax;
                q_mult *= __ldg(p.q_scale + static_cast<size_t>(bh) * nblk + qs / 128);
            }
            // FP8 factors of the next key tile (bf16: the scale alone).
            float nx_mult = q_mult, nx_lg = 0.0f, nx_inv = 1.0f;
            if constexpr (Cfg::FP8)
                fp8_tile_scales<Cfg>(p, sb0 + (tk.first * BN) / 128, q_mult, ivmax, nx_mult, nx_lg, nx_inv);
            float m = -INFINITY;   // reference maximum of the log2-scaled scores
            float l = 0.0f;        // running sum of exp2(score - m)
            bool first_tile = true;
            for (int j = tk.first; j >= 0; j = next_in<Cfg>(tk, j)) {
                bool wt = wait_phase(&bars->s_full[t], count & 1, abort_flag, p, SITE_SOFTMAX_S);
                if (!__all_sync(0xffffffffu, wt)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float mult = nx_mult;
                uint32_t sr[BN];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) tmem_ld32(s_tmem + c * 32, sr + c * 32);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) reg_fence32(sr + c * 32);

                const int kbase = j * BN;
                if (kbase < klo || kbase + BN - 1 > khi) {
#pragma unroll
                    for (int c = 0; c < BN; ++c) {
                        const int key = kbase + c;
                        if (key < klo || key > khi) sr[c] = __float_as_uint(-INFINITY);
                    }
                }
                // Row maximum: four independent chains of 3-input max.
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
                // Reference maximum m.  It moves only when the row maximum
                // exceeds it by more than RESCALE_LOG2 (so P <= 2^RESCALE_LOG2;
                // exact, since O and l share the reference), and then to the
                // row maximum plus RESCALE_HEADROOM.
                const float m_tile = mx * mult;
                float m_new = m;
                if (m_tile > m + Cfg::RESCALE_LOG2 || m == -INFINITY)
                    m_new = fmaxf(m, m_tile + Cfg::RESCALE_HEADROOM);
                // A row that has seen no visible key yet keeps m = -inf (so
                // that its first real scores set the reference, however
                // negative); its exponent reference is then 0 and its P is 0.
                const float m_use = m_new == -INFINITY ? 0.0f : m_new;
                const float alpha = ex2_approx(m - m_use);
                const float2 mult2 = make_float2(mult, mult);
                const float2 neg2 = make_float2(-m_use, -m_use);
                float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
                if constexpr (!Cfg::FP8) {
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
                        tmem_st16(s_tmem + c * 16, pk);
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
                        tmem_st16(s_tmem + c * 16, pk);
                    }
                    acc0 = __fadd2_rn(f16x2_to_float2(hs0), f16x2_to_float2(hs2));
                    acc1 = __fadd2_rn(f16x2_to_float2(hs1), f16x2_to_float2(hs3));
                    const float inv = nx_inv;
                    acc0.x *= inv; acc0.y *= inv; acc1.x *= inv; acc1.y *= inv;
                }
                const float rsum = (acc0.x + acc0.y) + (acc1.x + acc1.y);
                l = l * alpha + rsum;
                // Rescale the accumulator of the rows whose maximum moved.  The
                // commit that signalled S_t(j) also covers O_t += P_t V_{j-1}, so
                // O_t is stable here; the next P V waits for p_full below.
                // The whole row is loaded before one wait (one TMEM round trip
                // instead of one per 32 columns); S is dead by now.
                if (!first_tile && __any_sync(0xffffffffu, alpha != 1.0f)) {
                    uint32_t orr[D];
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) tmem_ld32(o_tmem + c * 32, orr + c * 32);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) reg_fence32(orr + c * 32);
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                    for (int x = 0; x < D; x += 2) {
                        const float2 v =
                            __fmul2_rn(make_float2(__uint_as_float(orr[x]), __uint_as_float(orr[x + 1])), a2);
                        orr[x] = __float_as_uint(v.x);
                        orr[x + 1] = __float_as_uint(v.y);
                    }
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) tmem_st32(o_tmem + c * 32, orr + c * 32);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars->p_full[t]);
                if constexpr (Cfg::FP8) {
                    const int jn = next_in<Cfg>(tk, j);
                    if (jn >= 0) {
                        fp8_tile_scales<Cfg>(p, sb0 + (jn * BN) / 128, q_mult, ivmax, nx_mult, nx_lg, nx_inv);
                        pin3(nx_mult, nx_lg, nx_inv);
                    }
                }
                m = m_new;
                first_tile = false;
                ++count;
            }
            if (!ok) break;
            {
                bool wt = wait_phase(&bars->o_full[t], qn & 1, abort_flag, p, SITE_SOFTMAX_O);
                ok = __all_sync(0xffffffffu, wt);
                ++qn;
            }
            if (!ok) break;
            tc_fence_after();
            // l = 0 only for a row that sees no key: O = 0, LSE = -inf.
            float out_mult = l > 0.0f ? 1.0f / l : 0.0f;
            if constexpr (Cfg::FP8) out_mult *= vmax * (1.0f / Cfg::P8_SCALE);
            if constexpr (Cfg::O_VIA_TMA) {
                // One 64-column box at a time: TMEM -> bf16 in registers -> this
                // warp's slot (row = lane, 16-byte chunk x at x ^ (lane & 7)) ->
                // TMA store of rows [row0, row0 + 32).  The conversion of a box
                // overlaps the store of the previous one reading the slot.
                const int row0 = qs + quad * 32;
                // (the slots sit right below the barriers: no extra live pointer)
                uint8_t* slot = reinterpret_cast<uint8_t*>(bars) - Cfg::EPI_BYTES + warp * Cfg::EPI_SLOT_BYTES;
#pragma unroll
                for (int cb = 0; cb < D / 64; ++cb) {
                    uint32_t orr[64];
                    tmem_ld32(o_tmem + cb * 64, orr);
                    tmem_ld32(o_tmem + cb * 64 + 32, orr + 32);
                    tmem_wait_ld();
                    reg_fence32(orr);
                    reg_fence32(orr + 32);
                    uint32_t pk[32];
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        pk[x] = pack_bf16x2(__uint_as_float(orr[2 * x]) * out_mult,
                                            __uint_as_float(orr[2 * x + 1]) * out_mult);
                    if (lane == 0) bulk_wait_group_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int x = 0; x < 8; ++x)
                        *reinterpret_cast<uint4*>(slot + lane * 128 + ((x ^ (lane & 7)) << 4)) =
                            make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && row0 < p.N) {
                        tma_store_4d(&tmap_o, slot, cb * 64, h, row0, b);
                        bulk_commit_group();
                    }
                }
            } else {
                const bool store = i < p.N;
                __nv_bfloat16* orow =
                    reinterpret_cast<__nv_bfloat16*>(p.o) + ((static_cast<size_t>(b) * p.N + i) * p.H + h) * D;
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
                        for (int x = 0; x < 4; ++x)
                            dst[x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
                    }
                }
            }
            if (i < p.N) p.lse[static_cast<size_t>(bh) * p.N + i] = (m + __log2f(l)) * 0.69314718055994530942f;
        }
        // The output stores have finished reading the slots (and written O)
        // before the CTA can exit.
        if constexpr (Cfg::O_VIA_TMA) {
            if (lane == 0) bulk_wait_group_all();
            __syncwarp();
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
