// FP8 prep on the tensor cores (block scales, with or without the Hadamard
// rotation), for head dims 64 and 128.  FlashAttention-3 deep-reading report
// §2.2 and §3.3: block quantisation, and incoherent processing that
// multiplies Q and K by M = diag(+-1) x Hadamard, which leaves Q K^T
// unchanged.
//
// The rotation of one 128-token block X (128 x d, bf16) is the product
// X (D H), and D H is a +-1 matrix, exact in bf16: one tcgen05 MMA chain per
// block (fp32 accumulation in tensor memory) replaces the d log d butterflies
// and their cross-lane shuffles.  Per block:
//   * TMA brings X into shared memory (128-byte swizzle, K-major; two stages,
//     so the next block's load overlaps this block's work);
//   * one thread issues the MMAs X (D H) into one of two tensor-memory
//     buffers, one block ahead of the epilogue;
//   * the 128 threads (thread r = token row r of the block) read their row
//     (tensor memory for rotated tensors, shared memory for the others),
//     scale it by 1/sqrt(d), reduce the block's amax, and write the e4m3
//     codes of row / (amax / 448) with the same correctly rounded quotient
//     as the CUDA-core prep.
// One launch may cover up to three tensors (Q, K, V): the blocks of all of
// them form one persistent work list (one CTA per SM, two independent
// 128-thread pipelines per CTA); each tensor says whether it is rotated.
#include <cuda_bf16.h>

#include <cstdint>

#include "fp8_prep.cuh"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kRows = 128;               // tokens per block (one scale)
constexpr int kGroups = 2;               // epilogue groups per CTA
constexpr int kGroupThreads = 128;       // one thread per token row of a block
// The producer warp (warp 8) leads a third warpgroup whose other warps idle:
// the register split (setmaxnreg) works per warpgroup.
constexpr int kThreads = (kGroups + 1) * 128;
constexpr int kLaunchRegs = 168;         // 65536 / 384, rounded down to 8
constexpr int kLowRegs = 56;             // the producer's warpgroup
constexpr int kHighRegs = 224;           // the epilogue warpgroups
static_assert(kHighRegs * kGroups * 128 + kLowRegs * 128 <= kLaunchRegs * kThreads, "register split");
constexpr int kSitePrepTcLoad = 0x92;    // status sites: the prep gave up waiting
constexpr int kSitePrepTcMma = 0x93;
constexpr int kSitePrepTcProducer = 0x94;

template <int D>
struct TcCfg {
    static constexpr int X_BYTES = kRows * D * 2;         // one bf16 block
    static constexpr int M_BYTES = D * D * 2;             // the signed Hadamard matrix (bf16)
    static constexpr int NCB = D / 64;                    // 64-element (128-byte) column boxes
    // Stages per group: loads run up to STAGES blocks ahead of the epilogue.
    static constexpr int STAGES = D == 128 ? 3 : 4;
    static constexpr int SMEM = 1024 + M_BYTES + kGroups * STAGES * X_BYTES;
    static constexpr int TMEM_COLS = kGroups * 2 * D;     // two fp32 accumulators per group
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

// Byte offset of element (row, col) of a bf16 tile of `rows` rows stored as
// 64-column boxes of 128-byte rows with the 128-byte swizzle (16-byte chunk
// j of row r sits at chunk j ^ (r mod 8)): the layout TMA writes for the
// attention tiles and the MMA descriptors read.
__device__ __forceinline__ uint32_t swz_offset(int row, int col, int rows) {
    const int box = col >> 6;
    const int byte = (col & 63) * 2;
    const int chunk = (byte >> 4) ^ (row & 7);
    return static_cast<uint32_t>(box * rows * 128 + row * 128 + chunk * 16 + (byte & 15));
}

// Non-blocking probe of an mbarrier phase (the producer polls several).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, unsigned long long limit,
                                             volatile int* abort_flag, int* status, int site) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (static_cast<unsigned long long>(clock64() - t0) > limit) {
            *abort_flag = 1;
            atomicCAS(status, 0, site);
            return false;
        }
    }
    return true;
}

// Barrier `id` among the `count` threads of one group that also ANDs a
// predicate over them.
__device__ __forceinline__ bool group_barrier_and(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// amax / 448 rounded to nearest (the block scale): Markstein's correction of
// the product with RN(1/448) gives the correctly rounded quotient for the
// normal-range values here, as the division would.
__device__ __forceinline__ float div448(float a) {
    constexpr float inv448 = 1.0f / 448.0f;
    const float q0 = a * inv448;
    const float rem = fmaf(-q0, 448.0f, a);
    return fmaf(rem, inv448, q0);
}

// One CTA per SM.  The CTA's blocks are g = blockIdx.x + j * gridDim.x; group
// w (threads 128 w .. 128 w + 127) takes j = w, w + 2, ...  The producer warp
// (warp 8) issues every TMA load and MMA of both groups, as soon as a stage
// or an accumulator is free, so the groups' threads only wait for results:
//   full[w][s]       load of stage s landed (transaction bytes)
//   stage_free[w][s] stage s read (its MMA done, or its rows read), 4 arrivals
//   mma_done[w][b]   X (D H) into accumulator b complete
//   tmem_free[w][b]  accumulator b read by the group, 4 arrivals
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fp8_prep_tc_kernel(const __grid_constant__ CUtensorMap m0, const __grid_constant__ CUtensorMap m1,
                       const __grid_constant__ CUtensorMap m2, const PrepTcParams p) {
    using C = TcCfg<D>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* mh = smem;                                  // D H, K-major rows n, columns k
    __shared__ uint64_t full[kGroups][S];
    __shared__ uint64_t stage_free[kGroups][S];
    __shared__ uint64_t mma_done[kGroups][2];
    __shared__ uint64_t tmem_free[kGroups][2];
    __shared__ uint32_t tmem_base;
    // Per group, per block parity (a warp can be at most one group barrier
    // ahead of another, so a block's maxima are never overwritten while read).
    __shared__ float warp_max[kGroups][2][4];
    __shared__ float sign[D];
    __shared__ int abort_flag;
    volatile int* abort_v = &abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = static_cast<int>(gridDim.x);
    const int nmine = p.total_blocks > static_cast<int>(blockIdx.x)
                          ? (p.total_blocks - static_cast<int>(blockIdx.x) + G - 1) / G
                          : 0;

    if (tid == 0) {
        for (int w = 0; w < kGroups; ++w) {
            for (int s = 0; s < S; ++s) {
                mbar_init(&full[w][s], 1);
                mbar_init(&stage_free[w][s], 4);
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(&mma_done[w][b], 1);
                mbar_init(&tmem_free[w][b], 4);
            }
        }
        abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&m0);
        tma_prefetch_desc(&m1);
        tma_prefetch_desc(&m2);
    }
    if (tid < D) sign[tid] = diag_sign(p.seed, tid);
    if (warp == 0) {
        tmem_alloc(&tmem_base, C::TMEM_COLS);
        tmem_relinquish();
    }
    __syncthreads();
    // D H in bf16: entry (n, k) = sign_k * (-1)^popcount(n & k) (Sylvester
    // Hadamard, unnormalised; 1/sqrt(d) is applied to the fp32 result), as
    // the B operand of X (D H): row n holds column n of D H.
    for (int c = tid; c < D * D / 8; c += kThreads) {
        const int n = c / (D / 8), k0 = (c % (D / 8)) * 8;
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int ka = k0 + 2 * q, kb = ka + 1;
            const float va = sign[ka] * ((__popc(n & ka) & 1) ? -1.0f : 1.0f);
            const float vb = sign[kb] * ((__popc(n & kb) & 1) ? -1.0f : 1.0f);
            w[q] = (va > 0.0f ? 0x3F80u : 0xBF80u) | ((vb > 0.0f ? 0x3F80u : 0xBF80u) << 16);
        }
        *reinterpret_cast<uint4*>(mh + swz_offset(n, k0, D)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // Block i of group g -> tensor, (batch, head), 128-row block.  The
    // tensor's fields are selected, not indexed (no copy of the parameters
    // to local memory).
    struct Blk {
        int t, b, h, blk, rotate, H;
        uint8_t* x8;
        float* scales;
    };
    auto decode = [&](int g, int i) {
        Blk r;
        int gl = static_cast<int>(blockIdx.x) + (2 * i + g) * G, t = 0;
        if (gl >= p.t[0].blocks) {
            gl -= p.t[0].blocks;
            t = 1;
            if (gl >= p.t[1].blocks) {
                gl -= p.t[1].blocks;
                t = 2;
            }
        }
        r.t = t;
        r.H = t == 0 ? p.t[0].H : (t == 1 ? p.t[1].H : p.t[2].H);
        r.rotate = t == 0 ? p.t[0].rotate : (t == 1 ? p.t[1].rotate : p.t[2].rotate);
        r.x8 = t == 0 ? p.t[0].x8 : (t == 1 ? p.t[1].x8 : p.t[2].x8);
        r.scales = t == 0 ? p.t[0].scales : (t == 1 ? p.t[1].scales : p.t[2].scales);
        const int bh = gl / p.nblk;
        r.blk = gl % p.nblk;
        r.b = bh / r.H;
        r.h = bh % r.H;
        return r;
    };
    auto group_blocks = [&](int g) { return (nmine - g + 1) / 2; };

    if (warp >= kGroups * 4) {
        regs_decrease<kLowRegs>();
        // ------------------------------------------------------------ producer
        if (warp == kGroups * 4 && lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int li[kGroups], mi[kGroups], ngr[kGroups];
            int ru0[kGroups], ru1[kGroups];     // rotated blocks issued into accumulator 0 / 1
#pragma unroll
            for (int g = 0; g < kGroups; ++g) {
                li[g] = mi[g] = 0;
                ngr[g] = group_blocks(g);
                ru0[g] = ru1[g] = 0;
            }
            auto load = [&](int g, int i) {
                const Blk k = decode(g, i);
                const int st = i % S;
                const CUtensorMap* mp = k.t == 0 ? &m0 : (k.t == 1 ? &m1 : &m2);
                uint8_t* dst = smem + C::M_BYTES + (g * S + st) * C::X_BYTES;
                mbar_arrive_expect_tx(&full[g][st], C::X_BYTES);
#pragma unroll
                for (int cb = 0; cb < C::NCB; ++cb)
                    tma_load_4d(dst + cb * (kRows * 128), mp, &full[g][st], cb * 64, k.h, k.blk * kRows, k.b, pol);
            };
            long long t_last = clock64();
            while (true) {
                bool progress = false, done = true;
#pragma unroll
                for (int g = 0; g < kGroups; ++g) {
                    // Loads: block li into its stage once the block S before it
                    // has released the stage.
                    if (li[g] < ngr[g] &&
                        (li[g] < S || mbar_test(&stage_free[g][li[g] % S], ((li[g] - S) / S) & 1))) {
                        load(g, li[g]);
                        ++li[g];
                        progress = true;
                    }
                    // MMAs, in block order: block mi once its load has landed
                    // and its accumulator has been read by the group.
                    if (mi[g] < ngr[g] && mi[g] < li[g]) {
                        const Blk k = decode(g, mi[g]);
                        if (!k.rotate) {
                            ++mi[g];
                            progress = true;
                        } else {
                            const int st = mi[g] % S, b = mi[g] & 1;
                            const int uses = b ? ru1[g] : ru0[g];
                            if (mbar_test(&full[g][st], (mi[g] / S) & 1) &&
                                (uses == 0 || mbar_test(&tmem_free[g][b], (uses - 1) & 1))) {
                                tc_fence_after();
                                constexpr uint32_t idesc = make_idesc(1u, 128, D, 0);
                                const uint64_t adesc = sdesc_swz<128>(
                                    smem_u32(smem + C::M_BYTES + (g * S + st) * C::X_BYTES), 16, 8 * 128);
                                const uint64_t bdesc = sdesc_swz<128>(smem_u32(mh), 16, 8 * 128);
                                const uint32_t dcol = tmem_base + (g * 2 + b) * D;
#pragma unroll
                                for (int kk = 0; kk < D / 16; ++kk) {
                                    const int byte_k = kk * 32;
                                    const uint32_t a_off = (byte_k / 128) * (kRows * 128) + (byte_k % 128);
                                    const uint32_t b_off = (byte_k / 128) * (D * 128) + (byte_k % 128);
                                    mma_f16_ss(dcol, adesc + (a_off >> 4), bdesc + (b_off >> 4), idesc,
                                               kk > 0 ? 1u : 0u);
                                }
                                mma_commit(&mma_done[g][b]);
                                if (b) ++ru1[g];
                                else ++ru0[g];
                                ++mi[g];
                                progress = true;
                            }
                        }
                    }
                    if (li[g] < ngr[g] || mi[g] < ngr[g]) done = false;
                }
                if (done) break;
                if (progress) {
                    t_last = clock64();
                } else {
                    // Nothing to issue: back off so the polls do not take issue
                    // slots from the epilogue warps of this sub-partition.
                    __nanosleep(64);
                    if (*abort_v) break;
                    if (static_cast<unsigned long long>(clock64() - t_last) > p.wait_limit) {
                        *abort_v = 1;
                        atomicCAS(p.status, 0, kSitePrepTcProducer);
                        break;
                    }
                }
            }
            // Teardown: every load this thread issued lands and every MMA it
            // committed completes before the CTA can free tensor memory.
            const long long t0 = clock64();
            const unsigned long long lim = p.wait_limit > 2000000000ull ? p.wait_limit : 2000000000ull;
#pragma unroll
            for (int g = 0; g < kGroups; ++g) {
                for (int i = li[g] > S ? li[g] - S : 0; i < li[g]; ++i)
                    while (!mbar_test(&full[g][i % S], (i / S) & 1))
                        if (static_cast<unsigned long long>(clock64() - t0) > lim) break;
                if (ru0[g] > 0)
                    while (!mbar_test(&mma_done[g][0], (ru0[g] - 1) & 1))
                        if (static_cast<unsigned long long>(clock64() - t0) > lim) break;
                if (ru1[g] > 0)
                    while (!mbar_test(&mma_done[g][1], (ru1[g] - 1) & 1))
                        if (static_cast<unsigned long long>(clock64() - t0) > lim) break;
            }
        }
        __syncwarp();
    } else {
        regs_increase<kHighRegs>();
        // ------------------------------------------------------------ epilogue groups
        const int grp = warp >> 2, gwarp = warp & 3, tw = tid & 127;
        const uint32_t bar_id = 1 + grp;
        const int ngrp = group_blocks(grp);
        const uint32_t lane_base = static_cast<uint32_t>(gwarp * 32) << 16;
        constexpr float inv_sqrt_d = D == 64 ? 0.125f : 0.08838834764831845f;
        int rot_seen[2] = {0, 0};           // rotated blocks consumed per accumulator
        bool ok = true;
        for (int i = 0; i < ngrp && ok; ++i) {
            const int s = i & 1;                    // accumulator (and maxima buffer)
            const int st = i % S;                   // stage
            const Blk k = decode(grp, i);
            float r[D];
            if (k.rotate) {
                const int uses = s ? rot_seen[1] : rot_seen[0];
                const bool w =
                    bounded_wait(&mma_done[grp][s], uses & 1, p.wait_limit, abort_v, p.status, kSitePrepTcMma);
                if (s) ++rot_seen[1];
                else ++rot_seen[0];
                if (!__all_sync(0xffffffffu, w)) ok = false;
                if (ok) {
                    tc_fence_after();
                    uint32_t* v = reinterpret_cast<uint32_t*>(r);
#pragma unroll
                    for (int c = 0; c < D / 32; ++c)
                        tmem_ld32(tmem_base + lane_base + (grp * 2 + s) * D + c * 32, v + c * 32);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) reg_fence32(v + c * 32);
                    // The accumulator and (its MMA being done) the stage are free.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&tmem_free[grp][s]);
                        mbar_arrive(&stage_free[grp][st]);
                    }
                    // "+ 0.0f" maps a -0 (an exact zero from cancelling signs) to +0,
                    // so that a zero encodes as the +0 code.
#pragma unroll
                    for (int e = 0; e < D; ++e) r[e] = fmaf(r[e], inv_sqrt_d, 0.0f);
                } else {
#pragma unroll
                    for (int e = 0; e < D; ++e) r[e] = 0.0f;
                }
            } else {
                // Not rotated: the row straight from the swizzled stage.
                const bool w =
                    bounded_wait(&full[grp][st], (i / S) & 1, p.wait_limit, abort_v, p.status, kSitePrepTcLoad);
                if (!__all_sync(0xffffffffu, w)) ok = false;
                const uint8_t* xrow = smem + C::M_BYTES + (grp * S + st) * C::X_BYTES;
#pragma unroll
                for (int c = 0; c < D / 8; ++c) {
                    const uint4 u = *reinterpret_cast<const uint4*>(xrow + swz_offset(tw, c * 8, kRows));
                    const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        r[c * 8 + 2 * q] = __uint_as_float(wv[q] << 16);
                        r[c * 8 + 2 * q + 1] = __uint_as_float(wv[q] & 0xFFFF0000u);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&stage_free[grp][st]);
            }
            // Row amax: eight independent chains of 3-input maxima (a single
            // chain would serialise D dependent operations).
            float am[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) am[c] = fmaxf(fabsf(r[2 * c]), fabsf(r[2 * c + 1]));
#pragma unroll
            for (int e = 16; e < D; e += 16) {
#pragma unroll
                for (int c = 0; c < 8; ++c) am[c] = fmax3(am[c], fabsf(r[e + 2 * c]), fabsf(r[e + 2 * c + 1]));
            }
            float amax = fmax3(fmax3(am[0], am[1], am[2]), fmax3(am[3], am[4], am[5]), fmaxf(am[6], am[7]));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            if (lane == 0) warp_max[grp][s][gwarp] = amax;
            ok = group_barrier_and(bar_id, kGroupThreads, ok);
            if (!ok) break;
            // Every thread takes the block's scale from the four warp maxima (the
            // same correctly rounded quotient everywhere).
            const float a = fmaxf(fmaxf(warp_max[grp][s][0], warp_max[grp][s][1]),
                                  fmaxf(warp_max[grp][s][2], warp_max[grp][s][3]));
            const float sc = a > 0.0f ? div448(a) : 1.0f;
            if (tw == 0) k.scales[(static_cast<size_t>(k.b) * k.H + k.h) * p.nblk + k.blk] = sc;
            const float inv = __frcp_rn(sc);
            const int n = k.blk * kRows + tw;
            if (n < p.N) {
                uint8_t* dst = k.x8 + ((static_cast<size_t>(k.b) * p.N + n) * k.H + k.h) * D;
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {
                    uint32_t w[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int e = c * 16 + q * 4;
                        w[q] = pack_e4m3x4(div_by_scale(r[e], sc, inv), div_by_scale(r[e + 1], sc, inv),
                                           div_by_scale(r[e + 2], sc, inv), div_by_scale(r[e + 3], sc, inv));
                    }
                    reinterpret_cast<uint4*>(dst)[c] = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int D>
cudaError_t launch_tc(const CUtensorMap* maps, const PrepTcParams& p, const PrepLaunch& L, cudaStream_t stream) {
    using C = TcCfg<D>;
    auto kernel = fp8_prep_tc_kernel<D>;
    // The register split assumes every thread is launched with kLaunchRegs
    // registers; a build with another count could make the increase wait
    // forever, so it is refused.
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, kernel);
    if (e != cudaSuccess) return e;
    if (attr.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    // One CTA per SM (it holds all of tensor memory at d = 128), persistent.
    const long long cap = L.num_sms;
    const unsigned grid = static_cast<unsigned>(p.total_blocks < cap ? p.total_blocks : cap);
    kernel<<<grid, kThreads, C::SMEM, stream>>>(maps[0], maps[1], maps[2], p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t run_fp8_prep_tc(const CUtensorMap* maps, const PrepTcParams& p, int d, const PrepLaunch& L,
                            cudaStream_t stream) {
    if (p.total_blocks <= 0) return cudaSuccess;
    switch (d) {
        case 64: return launch_tc<64>(maps, p, L, stream);
        case 128: return launch_tc<128>(maps, p, L, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
