// FP8 prep kernel: r = x D H_d / sqrt(d) (Q and K, mode 1), then per block
// of 128 tokens of one (batch, head): amax, scale = amax / 448, e4m3 codes
// of r / scale.  FlashAttention-3 deep-reading report §2.2 and §3.3 (block
// quantization; incoherent processing with M = diag(+-1) x Hadamard, O(d log d)).
//
// A CTA handles whole 128-token blocks of one head at a time, so the block
// amax is a CTA reduction and the data is read once and written once (the op
// is bound by device-memory bandwidth); the block's bf16 tile arrives in
// shared memory by TMA, double-buffered across the CTA's blocks.  A warp holds whole rows: lane l keeps elements
// [l*E, l*E + E) of a row, E = d / 32.  The Walsh-Hadamard butterflies with
// stride < E stay inside a thread; the wider ones pair lanes with shuffles.
// With RoPE (rotary position embedding; Su et al., "RoFormer", 2021) the
// row is first turned pair by pair with the caller's binary32 cos / sin
// tables (N, d/2): a' = a cos - b sin, b' = a sin + b cos, each product and
// sum rounded (no FMA), pairs (i, i + d/2) ("half-split": the partner sits
// 16 lanes away) or (2i, 2i + 1) ("interleaved": inside the thread).  This is
// the placement the report's §2.2 names: quantisation riding inside the
// memory-bound rotary-embedding pass.
// Mode 2 (one scale per tensor) runs three launches: block amax into
// `scales`, a one-CTA reduction that turns them into the tensor's scale,
// and the quantisation with that scale.
#include <cuda_bf16.h>

#include <cstdint>

#include "fp8_prep.cuh"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kBlockRows = 128;

enum Pass { kFused = 0, kAmaxOnly = 1, kApplyScale = 2 };
constexpr int kSitePrepLoad = 0x91;   // status site: the prep gave up waiting for a tile
enum Rope { kNoRope = 0, kRopeHalf = 1, kRopeInterleaved = 2 };

template <int K> struct FloatVec;
template <> struct FloatVec<1> { using T = float; };
template <> struct FloatVec<2> { using T = float2; };
template <> struct FloatVec<4> { using T = float4; };
template <> struct FloatVec<8> { using T = float4; };   // loaded as two float4

// K consecutive floats from a 4*K-byte aligned address.
template <int K>
__device__ __forceinline__ void load_floats(const float* __restrict__ p, float (&out)[K]) {
    if constexpr (K == 8) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p));
        const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
        out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
        out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
    } else {
        const typename FloatVec<K>::T v = __ldg(reinterpret_cast<const typename FloatVec<K>::T*>(p));
        const float* f = reinterpret_cast<const float*>(&v);
#pragma unroll
        for (int k = 0; k < K; ++k) out[k] = f[k];
    }
}

template <int E> struct RowLoad;
template <> struct RowLoad<2> { using T = uint32_t; };
template <> struct RowLoad<4> { using T = uint2; };
template <> struct RowLoad<8> { using T = uint4; };

// Persistent: CTA c takes the blocks c, c + G, c + 2G, ... (G = grid).  While
// it rotates and quantises one block (read from shared memory), the TMA
// brings the next block into the other of two stages, so the device-memory
// reads of the next block overlap the arithmetic and the stores of this one.
template <int D, int WARPS, int PASS, int ROPE>
__global__ void __launch_bounds__(WARPS * 32)
    fp8_prep_kernel(const __grid_constant__ CUtensorMap tmap_x, uint8_t* __restrict__ x8,
                    float* __restrict__ scales, int H, int N, int nblk, int total_blocks, int rotate,
                    unsigned long long seed, const float* __restrict__ rope_cos, const float* __restrict__ rope_sin,
                    unsigned long long wait_limit, int* status) {
    constexpr int E = D / 32;                     // elements per lane
    // table entries a lane needs per row: E (half-split) or E/2 (interleaved)
    constexpr int TE = ROPE == kRopeInterleaved ? E / 2 : E;
    constexpr int RPW = kBlockRows / WARPS;       // rows per warp
    constexpr int TILE_BYTES = kBlockRows * D * 2;
    using Raw = typename RowLoad<E>::T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t* stage_base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    __shared__ uint64_t full[2];
    __shared__ float warp_max[WARPS];
    __shared__ float block_scale;
    __shared__ int abort_flag;

    if (threadIdx.x == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmap_x);
    }
    __syncthreads();
    const uint64_t pol = l2_policy_evict_first();
    // Block index -> (batch * head, 128-row block); the tile's coordinates.
    auto issue_load = [&](int g, int s) {
        const int blk = g % nblk, bh = g / nblk;
        mbar_arrive_expect_tx(&full[s], TILE_BYTES);
        tma_load_4d(stage_base + s * TILE_BYTES, &tmap_x, &full[s], 0, bh % H, blk * kBlockRows, bh / H, pol);
    };
    if (threadIdx.x == 0 && static_cast<int>(blockIdx.x) < total_blocks) issue_load(blockIdx.x, 0);

    float sgn[E];
#pragma unroll
    for (int e = 0; e < E; ++e) sgn[e] = rotate ? diag_sign(seed, lane * E + e) : 1.0f;
    const int i0 = ROPE == kRopeHalf ? (lane & 15) * E : lane * (E / 2);   // first pair index

    int k = 0;          // blocks of this CTA so far
    int issued = 1;     // loads issued (the prologue's)
    for (int g = blockIdx.x; g < total_blocks; g += gridDim.x, ++k) {
        const int s = k & 1;
        const int blk = g % nblk;
        const int bh = g / nblk;
        const int b = bh / H, h = bh % H;
        const int n0 = blk * kBlockRows + warp * RPW;
        // The other stage was last read in the previous iteration (which ended
        // with a CTA barrier): refill it with the next block.
        if (threadIdx.x == 0 && g + static_cast<int>(gridDim.x) < total_blocks) {
            issue_load(g + gridDim.x, s ^ 1);
            ++issued;
        }
        // RoPE table entries of this lane's pairs: loaded up front for all
        // rows where the registers allow it (d <= 128), else row by row.
        constexpr bool PRELOAD = ROPE != kNoRope && D <= 128;
        constexpr int TROWS = PRELOAD ? RPW : 1;
        float tc[TROWS][TE], ts[TROWS][TE];
        auto load_table = [&](int rr, int slot) {
            const int n = min(n0 + rr, N - 1);
            load_floats<TE>(rope_cos + static_cast<size_t>(n) * (D / 2) + i0, tc[slot]);
            load_floats<TE>(rope_sin + static_cast<size_t>(n) * (D / 2) + i0, ts[slot]);
        };
        if constexpr (PRELOAD) {
#pragma unroll
            for (int rr = 0; rr < RPW; ++rr) load_table(rr, rr);
        }
        // Wait (bounded) for this block's tile.
        {
            bool ok = mbar_try_wait(&full[s], (k >> 1) & 1);
            if (!ok) {
                const long long t0 = clock64();
                while (!(ok = mbar_try_wait(&full[s], (k >> 1) & 1))) {
                    if (*static_cast<volatile int*>(&abort_flag)) break;
                    if (static_cast<unsigned long long>(clock64() - t0) > wait_limit) {
                        abort_flag = 1;
                        atomicCAS(status, 0, kSitePrepLoad);
                        break;
                    }
                }
            }
            if (!__syncthreads_and(ok ? 1 : 0)) break;
        }
        const uint8_t* tile = stage_base + s * TILE_BYTES;
        Raw raw[RPW];
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr)
            raw[rr] = *reinterpret_cast<const Raw*>(tile + ((warp * RPW + rr) * D + lane * E) * 2);

        float r[RPW][E];
        float amax = 0.0f;
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const __nv_bfloat162* pv = reinterpret_cast<const __nv_bfloat162*>(&raw[rr]);
#pragma unroll
            for (int q = 0; q < E / 2; ++q) {
                r[rr][2 * q] = __bfloat162float(pv[q].x);
                r[rr][2 * q + 1] = __bfloat162float(pv[q].y);
            }
            const int slot = PRELOAD ? rr : 0;
            if constexpr (ROPE != kNoRope && !PRELOAD) load_table(rr, 0);
            if constexpr (ROPE == kRopeHalf) {
                // lanes 0-15 hold the first halves a, lanes 16-31 the partners b
                const bool upper = lane >= 16;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float other = __shfl_xor_sync(0xffffffffu, r[rr][e], 16);
                    const float a = upper ? other : r[rr][e], bb = upper ? r[rr][e] : other;
                    const float c = tc[slot][e], sn = ts[slot][e];
                    r[rr][e] = upper ? __fadd_rn(__fmul_rn(a, sn), __fmul_rn(bb, c))
                                     : __fsub_rn(__fmul_rn(a, c), __fmul_rn(bb, sn));
                }
            } else if constexpr (ROPE == kRopeInterleaved) {
#pragma unroll
                for (int q = 0; q < E / 2; ++q) {
                    const float a = r[rr][2 * q], bb = r[rr][2 * q + 1];
                    const float c = tc[slot][q], sn = ts[slot][q];
                    r[rr][2 * q] = __fsub_rn(__fmul_rn(a, c), __fmul_rn(bb, sn));
                    r[rr][2 * q + 1] = __fadd_rn(__fmul_rn(a, sn), __fmul_rn(bb, c));
                }
            }
            if (rotate) {
#pragma unroll
                for (int e = 0; e < E; ++e) r[rr][e] *= sgn[e];
                // Butterflies inside the thread (strides 1 .. E/2).
#pragma unroll
                for (int st = 1; st < E; st <<= 1) {
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        if ((e & st) == 0) {
                            const float a = r[rr][e], c = r[rr][e + st];
                            r[rr][e] = a + c;
                            r[rr][e + st] = a - c;
                        }
                    }
                }
                // Butterflies across lanes (strides E .. D/2): the lower lane of
                // a pair keeps r + other, the upper one other - r, both as one
                // fused multiply-add by +-1 (the product is exact, so the result
                // is the plain sum / difference, rounded once).
#pragma unroll
                for (int ls = 1; ls < 32; ls <<= 1) {
                    const float pm = (lane & ls) ? -1.0f : 1.0f;
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float other = __shfl_xor_sync(0xffffffffu, r[rr][e], ls);
                        r[rr][e] = fmaf(r[rr][e], pm, other);
                    }
                }
                constexpr float inv_sqrt_d = D == 64 ? 0.125f : (D == 128 ? 0.08838834764831845f : 0.0625f);
                // "+ 0.0f" maps a -0 produced by a sign flip of an exact zero to +0,
                // so a zero always encodes as the +0 code; one fused multiply-add
                // rounds the exact product once, as the separate multiply would.
#pragma unroll
                for (int e = 0; e < E; ++e) r[rr][e] = fmaf(r[rr][e], inv_sqrt_d, 0.0f);
            }
#pragma unroll
            for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(r[rr][e]));
        }

        if constexpr (PASS != kApplyScale) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            if (lane == 0) warp_max[warp] = amax;
            __syncthreads();
            if (threadIdx.x == 0) {
                float a = warp_max[0];
#pragma unroll
                for (int w = 1; w < WARPS; ++w) a = fmaxf(a, warp_max[w]);
                if constexpr (PASS == kAmaxOnly) {
                    scales[static_cast<size_t>(bh) * nblk + blk] = a;
                } else {
                    const float sc = a > 0.0f ? __fdiv_rn(a, 448.0f) : 1.0f;
                    scales[static_cast<size_t>(bh) * nblk + blk] = sc;
                    block_scale = sc;
                }
            }
        } else {
            if (threadIdx.x == 0) block_scale = scales[static_cast<size_t>(bh) * nblk + blk];
        }
        __syncthreads();
        if constexpr (PASS != kAmaxOnly) {
            const float sc = block_scale;
            const float inv = __frcp_rn(sc);
#pragma unroll
            for (int rr = 0; rr < RPW; ++rr) {
                const int n = n0 + rr;
                if (n >= N) continue;
                uint8_t* dst = x8 + ((static_cast<size_t>(b) * N + n) * H + h) * D + lane * E;
                float y[E];
#pragma unroll
                for (int e = 0; e < E; ++e) y[e] = div_by_scale(r[rr][e], sc, inv);
                if constexpr (E == 2) {
                    uint16_t v;
                    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(v) : "f"(y[1]), "f"(y[0]));
                    *reinterpret_cast<uint16_t*>(dst) = v;
                } else if constexpr (E == 4) {
                    *reinterpret_cast<uint32_t*>(dst) = pack_e4m3x4(y[0], y[1], y[2], y[3]);
                } else {
                    uint2 v;
                    v.x = pack_e4m3x4(y[0], y[1], y[2], y[3]);
                    v.y = pack_e4m3x4(y[4], y[5], y[6], y[7]);
                    *reinterpret_cast<uint2*>(dst) = v;
                }
            }
        }
        // Every thread is done with this stage and with block_scale.
        __syncthreads();
    }
    // A load issued but never consumed (after a failed wait) lands before
    // the CTA exits.
    if (threadIdx.x == 0 && issued > k) {
        const long long t0 = clock64();
        const unsigned long long lim = wait_limit > 2000000000ull ? wait_limit : 2000000000ull;
        for (int j = k; j < issued; ++j)
            while (!mbar_try_wait(&full[j & 1], (j >> 1) & 1))
                if (static_cast<unsigned long long>(clock64() - t0) > lim) break;
    }
}

// Mode 2: the block maxima in `scales` -> one scale, written to every entry.
__global__ void __launch_bounds__(1024) per_tensor_scale_kernel(float* scales, long long count) {
    float a = 0.0f;
    for (long long i = threadIdx.x; i < count; i += blockDim.x) a = fmaxf(a, scales[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    __shared__ float wm[32];
    __shared__ float result;
    if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = a;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = 0.0f;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) m = fmaxf(m, wm[w]);
        result = m > 0.0f ? __fdiv_rn(m, 448.0f) : 1.0f;
    }
    __syncthreads();
    const float s = result;
    for (long long i = threadIdx.x; i < count; i += blockDim.x) scales[i] = s;
}

template <int D, int WARPS, int ROPE>
cudaError_t launch_prep(const CUtensorMap& map, void* x8, float* scales, int B, int H, int N, int mode,
                        unsigned long long seed, bool is_v, const float* rope_cos, const float* rope_sin,
                        const PrepLaunch& L, cudaStream_t stream) {
    const int nblk = (N + kBlockRows - 1) / kBlockRows;
    const long long blocks = static_cast<long long>(B) * H * nblk;
    if (blocks >= (1ll << 31)) return cudaErrorInvalidValue;
    auto* q8 = static_cast<uint8_t*>(x8);
    const int rotate = (mode == 1 && !is_v) ? 1 : 0;
    constexpr int smem = 2 * kBlockRows * D * 2 + 128;
    const dim3 block(WARPS * 32);
    const int total = static_cast<int>(blocks);
    auto run = [&](auto kernel, int rot) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        // Persistent grid: as many CTAs as can be resident at once (a CTA
        // that had to wait for a free SM would serialise its whole share).
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, WARPS * 32, smem);
        if (e != cudaSuccess) return e;
        const long long cap = static_cast<long long>(per_sm > 0 ? per_sm : 1) * L.num_sms;
        const dim3 grid(static_cast<unsigned>(blocks < cap ? blocks : cap));
        kernel<<<grid, block, smem, stream>>>(map, q8, scales, H, N, nblk, total, rot, seed, rope_cos, rope_sin,
                                              L.wait_limit, L.status);
        return cudaGetLastError();
    };
    if (mode != 2) return run(fp8_prep_kernel<D, WARPS, kFused, ROPE>, rotate);
    cudaError_t e = run(fp8_prep_kernel<D, WARPS, kAmaxOnly, ROPE>, 0);
    if (e != cudaSuccess) return e;
    per_tensor_scale_kernel<<<1, 1024, 0, stream>>>(scales, blocks);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return run(fp8_prep_kernel<D, WARPS, kApplyScale, ROPE>, 0);
}

template <int D, int WARPS>
cudaError_t launch_prep_any(const CUtensorMap& map, void* x8, float* scales, int B, int H, int N, int mode,
                            unsigned long long seed, bool is_v, const float* rope_cos, const float* rope_sin,
                            int rope, const PrepLaunch& L, cudaStream_t stream) {
    switch (rope) {
        case kNoRope:
            return launch_prep<D, WARPS, kNoRope>(map, x8, scales, B, H, N, mode, seed, is_v, nullptr, nullptr, L,
                                                  stream);
        case kRopeHalf:
            return launch_prep<D, WARPS, kRopeHalf>(map, x8, scales, B, H, N, mode, seed, is_v, rope_cos, rope_sin, L,
                                                    stream);
        case kRopeInterleaved:
            return launch_prep<D, WARPS, kRopeInterleaved>(map, x8, scales, B, H, N, mode, seed, is_v, rope_cos,
                                                           rope_sin, L, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t run_fp8_prep(const CUtensorMap& map, void* x8, float* scales, int B, int H, int N, int d, int mode,
                         unsigned long long sign_seed, bool is_v, const float* rope_cos, const float* rope_sin,
                         int rope, const PrepLaunch& L, cudaStream_t stream) {
    switch (d) {
        case 64:
            return launch_prep_any<64, 16>(map, x8, scales, B, H, N, mode, sign_seed, is_v, rope_cos, rope_sin, rope, L,
                                           stream);
        case 128:
            return launch_prep_any<128, 16>(map, x8, scales, B, H, N, mode, sign_seed, is_v, rope_cos, rope_sin, rope,
                                            L, stream);
        case 256:
            return launch_prep_any<256, 32>(map, x8, scales, B, H, N, mode, sign_seed, is_v, rope_cos, rope_sin, rope,
                                            L, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
