// C ABI of the fused exact-attention forward: argument checks, TMA tensor
// maps, dispatch to the kernel instantiations, status and error reporting.
// The declarations and the contract are in include/attn.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/attn.h"
#include "attn_bwd.cuh"
#include "attn_bwd_kernel.cuh"
#include "attn_launch.cuh"
#include "fp8_prep.cuh"

#include <algorithm>
#include <vector>

namespace attn {

bool causal_item_order(int nmb, int BH, int G, ItemOrder* order) {
    order->n = 0;
    const long long n = static_cast<long long>(nmb) * BH;
    if (n <= 0 || n > kOrderMax || G <= 0 || BH > 0xffff || nmb > 0xffff) return false;
    const int full = static_cast<int>((n / G) * G), rest = static_cast<int>(n) - full;
    struct It {
        int mb, bh;
    };
    // The `rest` lightest items, (query block ascending, head ascending)
    // positions below `rest`, form the last round; the rest, head by head
    // with the query block descending, make up the full rounds.
    std::vector<It> body, tail;
    body.reserve(static_cast<size_t>(full));
    for (int bh = 0; bh < BH; ++bh)
        for (int mb = nmb - 1; mb >= 0; --mb)
            if (static_cast<long long>(mb) * BH + bh >= rest) body.push_back({mb, bh});
    for (int mb = nmb - 1; mb >= 0; --mb)
        for (int bh = 0; bh < BH; ++bh)
            if (static_cast<long long>(mb) * BH + bh < rest) tail.push_back({mb, bh});
    auto heavier = [](const It& a, const It& b) { return a.mb > b.mb; };
    int k = 0;
    for (size_t r = 0; r < body.size(); r += static_cast<size_t>(G)) {
        auto first = body.begin() + static_cast<long>(r);
        auto last = body.begin() + static_cast<long>(std::min(body.size(), r + static_cast<size_t>(G)));
        std::stable_sort(first, last, heavier);     // heaviest first; heads ascending among equals
        for (auto x = first; x != last; ++x) order->e[k++] = static_cast<uint32_t>(x->mb) | (static_cast<uint32_t>(x->bh) << 16);
    }
    for (const It& x : tail) order->e[k++] = static_cast<uint32_t>(x.mb) | (static_cast<uint32_t>(x.bh) << 16);
    order->n = k;
    return k == n;
}

}  // namespace attn

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(ATTN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Device status word: first failing wait site of any kernel launched by the
// library (0 = none).  Its address is looked up once per device.
__device__ int g_attn_status;

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {};
std::mutex g_status_mutex;

constexpr unsigned long long kDefaultWaitLimit = 4000000000ull;   // ~2 s of SM clock
std::atomic<unsigned long long> g_wait_limit{kDefaultWaitLimit};

int status_ptr(int** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_status_mutex);
    if (!g_status_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_attn_status);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
        g_status_ptr[dev] = static_cast<int*>(ptr);
    }
    *out = g_status_ptr[dev];
    return ATTN_OK;
}

int g_sm_count[kMaxDevices] = {};

// Streaming multiprocessors of the current device (cached per device).
int sm_count(int* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_status_mutex);
    if (g_sm_count[dev] == 0) {
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(multiProcessorCount)");
        g_sm_count[dev] = n > 0 ? n : 1;
    }
    *out = g_sm_count[dev];
    return ATTN_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// (B, N, H, d) tensor viewed as 4-D {d, H, N, B}; box = one `swizzle`-byte
// column block (128, or 64 for 64-byte rows) of `rows` tokens of one head,
// with that swizzle (the layout the MMA shared-memory descriptors expect).
// Rows past N read as zero.
int make_map(CUtensorMap* map, const void* base, int B, int H, int N, int d, int elem_bytes, int rows,
             int swizzle = 128) {
    auto enc = encode_fn();
    if (!enc) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const CUtensorMapDataType dt =
        elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * elem_bytes, static_cast<cuuint64_t>(H) * d * elem_bytes,
                             static_cast<cuuint64_t>(N) * H * d * elem_bytes};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(swizzle / elem_bytes), 1, static_cast<cuuint32_t>(rows), 1};
    cuuint32_t estride[4] = {1, 1, 1, 1};
    CUresult r = enc(map, dt, 4, const_cast<void*>(base), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return ATTN_OK;
}

// bf16 (B, N, H, d) tensor as 4-D {d, H, N, B}; box = whole rows (d
// elements) of 128 tokens of one head, no swizzle: the FP8 prep's tile.
int make_row_map(CUtensorMap* map, const void* base, int B, int H, int N, int d) {
    auto enc = encode_fn();
    if (!enc) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(H) * d * 2,
                             static_cast<cuuint64_t>(N) * H * d * 2};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(d), 1, 128, 1};
    cuuint32_t estride[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estride,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled (rows) failed (CUresult %d)", static_cast<int>(r));
    return ATTN_OK;
}

// Everything the prep launch needs besides its arguments.
int prep_launch(const void* x, int B, int H, int N, int d, CUtensorMap* map, attn::PrepLaunch* L) {
    int rc = make_row_map(map, x, B, H, N, d);
    if (rc != ATTN_OK) return rc;
    if ((rc = sm_count(&L->num_sms)) != ATTN_OK) return rc;
    if ((rc = status_ptr(&L->status)) != ATTN_OK) return rc;
    L->wait_limit = g_wait_limit.load();
    return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The tensor-core prep (modes 0 and 1 at d = 64 and 128) of up to three bf16
// (B, N, H_i, d) tensors in one launch: x[i] -> codes x8[i], block scales
// scales[i]; rotate[i] = 1 multiplies tensor i by diag(+-1) x Hadamard.
int prep_tc(int n, const void* const* x, void* const* x8, float* const* scales, const int* Hs, const int* rotate,
            int B, int N, int d, unsigned long long sign_seed, cudaStream_t stream) {
    CUtensorMap maps[3];
    attn::PrepTcParams p{};
    p.N = N;
    p.nblk = (N + 127) / 128;
    long long total = 0;
    for (int i = 0; i < 3; ++i) {
        const int src = i < n ? i : 0;     // unused slots repeat tensor 0's map, with no blocks
        int rc = make_map(&maps[i], x[src], B, Hs[src], N, d, 2, 128, 128);
        if (rc != ATTN_OK) return rc;
        p.t[i].x8 = static_cast<uint8_t*>(x8[src]);
        p.t[i].scales = scales[src];
        p.t[i].H = Hs[src];
        p.t[i].rotate = rotate[src];
        const long long blocks = i < n ? static_cast<long long>(B) * Hs[i] * p.nblk : 0;
        p.t[i].blocks = static_cast<int>(blocks);
        total += blocks;
    }
    if (total >= (1ll << 31)) return fail(ATTN_ERR_INVALID_ARG, "problem too large for one launch");
    p.total_blocks = static_cast<int>(total);
    p.seed = sign_seed;
    attn::PrepLaunch L;
    int rc = sm_count(&L.num_sms);
    if (rc != ATTN_OK) return rc;
    if ((rc = status_ptr(&L.status)) != ATTN_OK) return rc;
    L.wait_limit = g_wait_limit.load();
    p.wait_limit = L.wait_limit;
    p.status = L.status;
    cudaError_t e = attn::run_fp8_prep_tc(maps, p, d, L, stream);
    if (e != cudaSuccess) return cuda_fail(e, "FP8 prep launch");
    return ATTN_OK;
}

int check_common(const void* q, const void* k, const void* v, const void* o, const float* lse, int B, int H, int N,
                 int d, int window) {
    if (B < 0 || H < 0 || N < 0) return fail(ATTN_ERR_INVALID_ARG, "negative size (B=%d H=%d N=%d)", B, H, N);
    if (d != 64 && d != 128 && d != 256) return fail(ATTN_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128, 256)", d);
    if (window < 0) return fail(ATTN_ERR_INVALID_ARG, "window %d < 0", window);
    if (static_cast<long long>(B) * H * N == 0) return ATTN_OK;
    if (!q || !k || !v || !o || !lse) return fail(ATTN_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return fail(ATTN_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    const long long items = static_cast<long long>(B) * H * ((N + 127) / 128);
    if (items >= (1ll << 31)) return fail(ATTN_ERR_INVALID_ARG, "problem too large for one launch");
    return ATTN_OK;
}

float resolve_scale(float scale, int d) {
    if (!(scale > 0.0f) || !std::isfinite(scale)) scale = 1.0f / std::sqrt(static_cast<float>(d));
    return scale;
}

int launch_forward(bool fp8, const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv,
                   int N, int d, int causal, float scale, int window, const float* qs, const float* ks, const float* vs,
                   void* stream, const uint8_t* block_mask = nullptr) {
    attn::FwdGeometry g;
    cudaError_t (*run)(const attn::FwdMaps&, const attn::FwdParams&, int, cudaStream_t) = nullptr;
    if (block_mask) {
        if (d == 64) {
            g = attn::geom_sparse_d64();
            run = attn::run_fwd_sparse_d64;
        } else if (d == 128) {
            g = attn::geom_sparse_d128();
            run = attn::run_fwd_sparse_d128;
        } else {
            g = attn::geom_sparse_d256();
            run = attn::run_fwd_sparse_d256;
        }
    } else if (fp8) {
        if (d == 128) {
            g = attn::geom_fp8_d128();
            run = attn::run_fwd_fp8_d128;
        } else if (d == 64) {
            g = attn::geom_fp8_d64();
            run = attn::run_fwd_fp8_d64;
        } else if (d == 256) {
            g = attn::geom_fp8_d256();
            run = attn::run_fwd_fp8_d256;
        } else {
            return fail(ATTN_ERR_UNSUPPORTED, "attn_fwd_fp8 supports head_dim 64, 128 and 256 (got %d)", d);
        }
    } else if (d == 64) {
        g = attn::geom_bf16_d64();
        run = attn::run_fwd_bf16_d64;
    } else if (d == 128) {
        g = attn::geom_bf16_d128();
        run = attn::run_fwd_bf16_d128;
    } else {
        g = attn::geom_bf16_d256();
        run = attn::run_fwd_bf16_d256;
    }
    attn::FwdMaps maps;
    int rc;
    if ((rc = make_map(&maps.q, q, B, H, N, d, g.elem_bytes, 128, g.swizzle)) != ATTN_OK) return rc;
    if ((rc = make_map(&maps.k, k, B, Hkv, N, d, g.elem_bytes, g.bn, g.swizzle)) != ATTN_OK) return rc;
    if ((rc = make_map(&maps.v, v, B, Hkv, N, d, g.elem_bytes, g.bn, g.swizzle)) != ATTN_OK) return rc;
    if ((rc = make_map(&maps.o, o, B, H, N, d, 2, 32, 128)) != ATTN_OK) return rc;
    attn::FwdParams p{};
    p.o = o;
    p.lse = lse;
    p.q_scale = qs;
    p.k_scale = ks;
    p.v_scale = vs;
    p.B = B;
    p.H = H;
    p.N = N;
    p.group = H / Hkv;
    p.causal = causal ? 1 : 0;
    p.window = window;
    p.scale_log2 = resolve_scale(scale, d) * 1.4426950408889634f;
    p.n_mblocks = (N + g.nq * 128 - 1) / (g.nq * 128);
    p.block_mask = block_mask;
    p.n_tb = (N + 127) / 128;
    p.wait_limit = g_wait_limit.load();
    if ((rc = status_ptr(&p.status)) != ATTN_OK) return rc;
    int sms = 0;
    if ((rc = sm_count(&sms)) != ATTN_OK) return rc;
    // Causal launches of the d = 128 kernels without grouped heads take their
    // work order from the launch parameters (copied at the launch, so the
    // buffer is free again when run() returns).  With grouped heads several
    // query heads already share each K/V head; the order then only crowds
    // more CTAs onto the same tiles.
    static thread_local attn::ItemOrder order;
    if (causal && !block_mask && d == 128 && Hkv == H) {
        const long long units = static_cast<long long>(p.n_mblocks) * B * H;
        const int G = static_cast<int>(units < sms ? units : sms);
        if (attn::causal_item_order(p.n_mblocks, B * H, G, &order)) maps.order = &order;
    }
    cudaError_t e = run(maps, p, sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, block_mask ? "attn_fwd_sparse launch" : (fp8 ? "attn_fwd_fp8 launch" : "attn_fwd launch"));
    return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_fwd_work_order(int n_mblocks, int BH, int grid, unsigned int* out, int capacity) {
    if (out == nullptr || n_mblocks <= 0 || BH <= 0 || grid <= 0) return 0;
    static thread_local attn::ItemOrder order;
    if (!attn::causal_item_order(n_mblocks, BH, grid, &order) || order.n > capacity) return 0;
    for (int i = 0; i < order.n; ++i) out[i] = order.e[i];
    return order.n;
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
             int causal, float scale, int window, void* stream) {
    return attn_fwd_gqa(q, k, v, o, lse, B, H, H, N, d, causal, scale, window, stream);
}

int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N,
                 int d, int causal, float scale, int window, void* stream) {
    g_err[0] = '\0';
    int rc = check_common(q, k, v, o, lse, B, H, N, d, window);
    if (rc != ATTN_OK) return rc;
    if (H_kv <= 0 || H % H_kv != 0)
        return fail(ATTN_ERR_INVALID_ARG, "key/value heads (%d) must divide query heads (%d)", H_kv, H);
    if (static_cast<long long>(B) * H * N == 0) return ATTN_OK;
    return launch_forward(false, q, k, v, o, lse, B, H, H_kv, N, d, causal, scale, window, nullptr, nullptr,
                          nullptr, stream);
}

int attn_fwd_fp8(const void* q8, const void* k8, const void* v8, void* o, float* lse, int B, int H, int N, int d,
                 int causal, float scale, int window, const float* q_scale, const float* k_scale,
                 const float* v_scale, void* stream) {
    return attn_fwd_fp8_gqa(q8, k8, v8, o, lse, B, H, H, N, d, causal, scale, window, q_scale, k_scale, v_scale,
                            stream);
}

int attn_fwd_fp8_gqa(const void* q8, const void* k8, const void* v8, void* o, float* lse, int B, int H, int H_kv,
                     int N, int d, int causal, float scale, int window, const float* q_scale, const float* k_scale,
                     const float* v_scale, void* stream) {
    g_err[0] = '\0';
    int rc = check_common(q8, k8, v8, o, lse, B, H, N, d, window);
    if (rc != ATTN_OK) return rc;
    if (H_kv <= 0 || H % H_kv != 0)
        return fail(ATTN_ERR_INVALID_ARG, "key/value heads (%d) must divide query heads (%d)", H_kv, H);
    if (static_cast<long long>(B) * H * N == 0) return ATTN_OK;
    if (d != 64 && d != 128 && d != 256)
        return fail(ATTN_ERR_UNSUPPORTED, "attn_fwd_fp8 supports head_dim 64, 128 and 256 (got %d)", d);
    if (!q_scale || !k_scale || !v_scale) return fail(ATTN_ERR_INVALID_ARG, "null scale pointer");
    return launch_forward(true, q8, k8, v8, o, lse, B, H, H_kv, N, d, causal, scale, window, q_scale, k_scale,
                          v_scale, stream);
}

int attn_fp8_prep(const void* x, void* x8, float* scales, int B, int H, int N, int d, int block_rows, int mode,
                  unsigned long long sign_seed, int is_v, void* stream) {
    g_err[0] = '\0';
    if (B < 0 || H < 0 || N < 0) return fail(ATTN_ERR_INVALID_ARG, "negative size (B=%d H=%d N=%d)", B, H, N);
    if (d != 64 && d != 128 && d != 256) return fail(ATTN_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128, 256)", d);
    if (block_rows != 128) return fail(ATTN_ERR_UNSUPPORTED, "block_rows must be 128 (got %d)", block_rows);
    if (mode < 0 || mode > 2) return fail(ATTN_ERR_INVALID_ARG, "mode %d (0, 1 or 2)", mode);
    if (static_cast<long long>(B) * H * N == 0) return ATTN_OK;
    if (!x || !x8 || !scales) return fail(ATTN_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(x) || !aligned16(x8) || !aligned16(scales))
        return fail(ATTN_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if ((mode == 0 || mode == 1) && d <= 128) {
        // The rotation as a tensor-core product.
        const int rot = (mode == 1 && !is_v) ? 1 : 0;
        return prep_tc(1, &x, &x8, &scales, &H, &rot, B, N, d, sign_seed, static_cast<cudaStream_t>(stream));
    }
    CUtensorMap map;
    attn::PrepLaunch L;
    int rc = prep_launch(x, B, H, N, d, &map, &L);
    if (rc != ATTN_OK) return rc;
    cudaError_t e = attn::run_fp8_prep(map, x8, scales, B, H, N, d, mode, sign_seed, is_v != 0, nullptr, nullptr, 0, L,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "attn_fp8_prep launch");
    return ATTN_OK;
}

int attn_fp8_prep_qkv(const void* q, const void* k, const void* v, void* q8, void* k8, void* v8, float* q_scale,
                      float* k_scale, float* v_scale, int B, int H, int H_kv, int N, int d, int mode,
                      unsigned long long sign_seed, void* stream) {
    g_err[0] = '\0';
    if (B < 0 || H < 0 || N < 0) return fail(ATTN_ERR_INVALID_ARG, "negative size (B=%d H=%d N=%d)", B, H, N);
    if (d != 64 && d != 128 && d != 256) return fail(ATTN_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128, 256)", d);
    if (mode < 0 || mode > 2) return fail(ATTN_ERR_INVALID_ARG, "mode %d (0, 1 or 2)", mode);
    if (H_kv <= 0 || H % H_kv != 0)
        return fail(ATTN_ERR_INVALID_ARG, "key/value heads (%d) must divide query heads (%d)", H_kv, H);
    if (static_cast<long long>(B) * H * N == 0) return ATTN_OK;
    const void* x[3] = {q, k, v};
    void* x8[3] = {q8, k8, v8};
    float* sc[3] = {q_scale, k_scale, v_scale};
    for (int i = 0; i < 3; ++i) {
        if (!x[i] || !x8[i] || !sc[i]) return fail(ATTN_ERR_INVALID_ARG, "null pointer");
        if (!aligned16(x[i]) || !aligned16(x8[i]) || !aligned16(sc[i]))
            return fail(ATTN_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    }
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((mode == 0 || mode == 1) && d <= 128) {
        const int Hs[3] = {H, H_kv, H_kv};
        const int rot[3] = {mode == 1 ? 1 : 0, mode == 1 ? 1 : 0, 0};
        return prep_tc(3, x, x8, sc, Hs, rot, B, N, d, sign_seed, s);
    }
    // Head dim 256 and the per-tensor mode: one launch per tensor.
    int rc = attn_fp8_prep(q, q8, q_scale, B, H, N, d, 128, mode, sign_seed, 0, stream);
    if (rc == ATTN_OK) rc = attn_fp8_prep(k, k8, k_scale, B, H_kv, N, d, 128, mode, sign_seed, 0, stream);
    if (rc == ATTN_OK) rc = attn_fp8_prep(v, v8, v_scale, B, H_kv, N, d, 128, mode, sign_seed, 1, stream);
    return rc;
}

int attn_fp8_prep_rope(const void* x, void* x8, float* scales, const float* rope_cos, const float* rope_sin,
                       int B, int H, int N, int d, int block_rows, int mode, unsigned long long sign_seed,
                       int interleaved, void* stream) {
    g_err[0] = '\0';
    if (B < 0 || H < 0 || N < 0) return fail(ATTN_ERR_INVALID_ARG, "negative size (B=%d H=%d N=%d)", B, H, N);
    if (d != 64 && d != 128 && d != 256) return fail(ATTN_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128, 256)", d);
    if (block_rows != 128) return fail(ATTN_ERR_UNSUPPORTED, "block_rows must be 128 (got %d)", block_rows);
    if (mode < 0 || mode > 2) return fail(ATTN_ERR_INVALID_ARG, "mode %d (0, 1 or 2)", mode);
    if (static_cast<long long>(B) * H * N == 0) return ATTN_OK;
    if (!x || !x8 || !scales || !rope_cos || !rope_sin) return fail(ATTN_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(x) || !aligned16(x8) || !aligned16(scales) || !aligned16(rope_cos) || !aligned16(rope_sin))
        return fail(ATTN_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    CUtensorMap map;
    attn::PrepLaunch L;
    int rc = prep_launch(x, B, H, N, d, &map, &L);
    if (rc != ATTN_OK) return rc;
    cudaError_t e = attn::run_fp8_prep(map, x8, scales, B, H, N, d, mode, sign_seed, false, rope_cos, rope_sin,
                                       interleaved ? 2 : 1, L, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "attn_fp8_prep_rope launch");
    return ATTN_OK;
}

int attn_fwd_sparse(const void* q, const void* k, const void* v, void* o, float* lse, const unsigned char* block_mask,
                    int B, int H, int H_kv, int N, int d, int causal, float scale, int window, void* stream) {
    g_err[0] = '\0';
    int rc = check_common(q, k, v, o, lse, B, H, N, d, window);
    if (rc != ATTN_OK) return rc;
    if (H_kv <= 0 || H % H_kv != 0)
        return fail(ATTN_ERR_INVALID_ARG, "key/value heads (%d) must divide query heads (%d)", H_kv, H);
    if (static_cast<long long>(B) * H * N == 0) return ATTN_OK;
    if (!block_mask) return fail(ATTN_ERR_INVALID_ARG, "null block mask");
    return launch_forward(false, q, k, v, o, lse, B, H, H_kv, N, d, causal, scale, window, nullptr, nullptr, nullptr,
                          stream, block_mask);
}

size_t attn_bwd_workspace_size(int B, int H, int N, int d) {
    if (B < 0 || H < 0 || N < 0 || d <= 0) return 0;
    return static_cast<size_t>(attn::bwd_workspace(B, H, N, d).bytes);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
             void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int H_kv, int N,
             int d, int causal, float scale, int window, void* stream) {
    g_err[0] = '\0';
    int rc = check_common(q, k, v, o, lse, B, H, N, d, window);
    if (rc != ATTN_OK) return rc;
    if (d != 128 && d != 64) return fail(ATTN_ERR_UNSUPPORTED, "attn_bwd supports head_dim 64 and 128 (got %d)", d);
    if (H_kv <= 0 || H % H_kv != 0)
        return fail(ATTN_ERR_INVALID_ARG, "key/value heads (%d) must divide query heads (%d)", H_kv, H);
    if (static_cast<long long>(B) * H * N == 0) return ATTN_OK;
    if (!dout || !dq || !dk || !dv || !workspace) return fail(ATTN_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return fail(ATTN_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(ATTN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    const attn::BwdWorkspace ws = attn::bwd_workspace(B, H, N, d);
    if (workspace_bytes < static_cast<size_t>(ws.bytes))
        return fail(ATTN_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %lld bytes needed",
                    workspace_bytes, ws.bytes);
    attn::BwdMaps maps;
    const int qrows = attn::bwd_query_rows(d);
    if ((rc = make_map(&maps.q, q, B, H, N, d, 2, qrows)) != ATTN_OK) return rc;
    if ((rc = make_map(&maps.dout, dout, B, H, N, d, 2, qrows)) != ATTN_OK) return rc;
    if ((rc = make_map(&maps.k, k, B, H_kv, N, d, 2, 128)) != ATTN_OK) return rc;
    if ((rc = make_map(&maps.v, v, B, H_kv, N, d, 2, 128)) != ATTN_OK) return rc;
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    attn::BwdParams p{};
    p.lse2 = reinterpret_cast<const float*>(wsb + ws.off_lse2);
    p.dvec = reinterpret_cast<const float*>(wsb + ws.off_dvec);
    p.dq_acc = reinterpret_cast<float*>(wsb + ws.off_dq);
    p.dk = dk;
    p.dv = dv;
    p.B = B;
    p.H = H;
    p.H_kv = H_kv;
    p.N = N;
    p.N_pad = ws.n_pad;
    p.group = H / H_kv;
    p.causal = causal ? 1 : 0;
    p.window = window;
    p.scale = resolve_scale(scale, d);
    p.scale_log2 = p.scale * 1.4426950408889634f;
    p.n_kblocks = (N + 127) / 128;
    p.wait_limit = g_wait_limit.load();
    if ((rc = status_ptr(&p.status)) != ATTN_OK) return rc;
    cudaError_t e = attn::run_bwd(d, maps, p, o, dout, lse, dq, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "attn_bwd launch");
    return ATTN_OK;
}

int attn_device_status(void* stream, int* site) {
    g_err[0] = '\0';
    if (site) *site = 0;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int* ptr = nullptr;
    int rc = status_ptr(&ptr);
    if (rc != ATTN_OK) return rc;
    int value = 0;
    e = cudaMemcpy(&value, ptr, sizeof value, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
    if (value != 0) {
        const int zero = 0;
        e = cudaMemcpy(ptr, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
        if (site) *site = value;
        return fail(ATTN_ERR_DEVICE_TIMEOUT, "a kernel gave up waiting at site 0x%x", value);
    }
    return ATTN_OK;
}

int attn_set_wait_limit(unsigned long long cycles) {
    g_err[0] = '\0';
    g_wait_limit.store(cycles ? cycles : kDefaultWaitLimit);
    return ATTN_OK;
}

const char* attn_last_error_string(void) { return g_err; }

}  // extern "C"

// ---------------------------------------------------------------------------
// attn_bwd_noalloc: the backward for callers that cannot allocate device
// memory (see include/attn.h).  Its scratch -- the LSE / D rows and the
// float32 dQ accumulator that attn_bwd keeps in the caller's workspace -- is
// this file-scope array, created once per device when the library's device
// code is loaded there and held until the process exits.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(256) << 20;   // 256 MiB
static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of g_bwd_scratch on the current device (host code may not
// use the array's name as a device address).  Looked up once per device.
int scratch_ptr(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_bwd_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(backward scratch)");
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return ATTN_OK;
}

}  // namespace

extern "C" {

size_t attn_bwd_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, int B, int H, int H_kv, int N, int d, int causal, float scale,
                     int window, void* stream) {
    g_err[0] = '\0';
    if (B < 0 || H < 0 || N < 0) return fail(ATTN_ERR_INVALID_ARG, "negative size (B=%d H=%d N=%d)", B, H, N);
    if ((d == 128 || d == 64) && static_cast<long long>(B) * H * N > 0) {
        const size_t need = attn_bwd_workspace_size(B, H, N, d);
        if (need > kNoAllocScratchBytes)
            return fail(ATTN_ERR_INVALID_ARG,
                        "attn_bwd_noalloc: this problem needs %zu bytes of scratch, more than the built-in %zu "
                        "(4 * B * H * ceil(N / 128) * 128 * (d + 2) bytes must fit); use attn_bwd with a workspace",
                        need, kNoAllocScratchBytes);
    }
    void* scratch = nullptr;
    if (static_cast<long long>(B) * H * N > 0) {
        const int rc = scratch_ptr(&scratch);
        if (rc != ATTN_OK) return rc;
    }
    // The prep launch of attn_bwd rewrites every scratch entry the call reads
    // (it zeroes the dQ accumulator), so nothing left by an earlier call leaks in.
    return attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, scratch, kNoAllocScratchBytes, B, H, H_kv, N, d, causal, scale,
                    window, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// attn_fwd_host: the forward on host buffers (see include/attn.h).  Chunks of
// whole sequences go through two device staging slots; per chunk c (slot
// c % 2, counted per device across calls):
//   h2d stream : wait freed[slot] (the D2H of the chunk that used the slot
//                before), copy Q, K, V in, record loaded[slot]
//   comp stream: wait loaded[slot], forward, record computed[slot]
//   d2h stream : wait computed[slot], copy O, LSE out, record freed[slot]
// so the copies in one direction overlap the forward and the copies in the
// other direction of the neighbouring chunks.

namespace {

constexpr int kHostChunks = 4;   // chunks per call (at most B)

struct HostPipe {
    cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
    cudaEvent_t entry = nullptr, done = nullptr;
    cudaEvent_t loaded[2] = {}, computed[2] = {}, freed[2] = {};
    unsigned long long chunks = 0;
    const void* last_ws = nullptr;   // staging layout of the previous call
    size_t last_slot = 0;
    bool ready = false;
};

HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mutex;   // guards g_pipe and the order of the enqueued work

// Called with g_pipe_mutex held.
int host_pipe(HostPipe** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    HostPipe& P = g_pipe[dev];
    if (!P.ready) {
        cudaStream_t* streams[3] = {&P.h2d, &P.comp, &P.d2h};
        for (cudaStream_t* s : streams) {
            if (*s) continue;
            e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreateWithFlags");
        }
        cudaEvent_t* events[8] = {&P.entry, &P.done, &P.loaded[0], &P.loaded[1],
                                  &P.computed[0], &P.computed[1], &P.freed[0], &P.freed[1]};
        for (cudaEvent_t* ev : events) {
            if (*ev) continue;
            e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
            if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreateWithFlags");
        }
        P.ready = true;
    }
    *out = &P;
    return ATTN_OK;
}

// Staging layout of one slot: the chunk's inputs, outputs and the scratch
// its compute step uses, each part 256-byte aligned.  Part sizes are given
// per sequence; the batch dimension is outermost in every host tensor.
struct Staging {
    long long cb = 0;                  // sequences per chunk
    int n_in = 0, n_out = 0;
    size_t in_seq[6] = {}, out_seq[3] = {};
    size_t in_off[6] = {}, out_off[3] = {}, scratch_off = 0, slot = 0;
};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

bool staging(int B, const size_t* in_seq, int n_in, const size_t* out_seq, int n_out, const size_t* scratch_seq,
             int n_scratch, Staging* L) {
    if (B <= 0) return false;
    const long long nch = B < kHostChunks ? B : kHostChunks;
    L->cb = (B + nch - 1) / nch;
    const size_t cb = static_cast<size_t>(L->cb);
    L->n_in = n_in;
    L->n_out = n_out;
    size_t off = 0;
    for (int x = 0; x < n_in; ++x) { L->in_seq[x] = in_seq[x]; L->in_off[x] = off; off += up256(cb * in_seq[x]); }
    for (int x = 0; x < n_out; ++x) { L->out_seq[x] = out_seq[x]; L->out_off[x] = off; off += up256(cb * out_seq[x]); }
    L->scratch_off = off;
    for (int x = 0; x < n_scratch; ++x) off += up256(cb * scratch_seq[x]);
    L->slot = off;
    return true;
}

// The forward's parts: Q, K, V in; O, LSE out.
bool fwd_staging(int B, int H, int H_kv, int N, int d, const size_t* scratch_seq, int n_scratch, Staging* L) {
    if (H <= 0 || H_kv <= 0 || N <= 0 || d <= 0) return false;
    const size_t q_seq = static_cast<size_t>(N) * H * d * 2, kv_seq = static_cast<size_t>(N) * H_kv * d * 2;
    const size_t in[3] = {q_seq, kv_seq, kv_seq}, out[2] = {q_seq, static_cast<size_t>(H) * N * 4};
    return staging(B, in, 3, out, 2, scratch_seq, n_scratch, L);
}

// Runs the chunks of one call through the staging slots (see above).
// compute(nb, slot_base, stream) queues the chunk's work on `stream`.
template <class Compute>
int host_pipeline(const void* const* in, void* const* out, int B, const Staging& L, void* workspace,
                  size_t workspace_bytes, void* stream, const char* who, Compute&& compute) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < 2 * L.slot)
        return fail(ATTN_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned and at least %zu bytes (got %zu)",
                    who, 2 * L.slot, workspace_bytes);
    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    HostPipe* P = nullptr;
    int rc = host_pipe(&P);
    if (rc != ATTN_OK) return rc;
    const cudaStream_t user = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaEventRecord(P->entry, user);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(P->h2d, P->entry, 0);
    if (e != cudaSuccess) return cuda_fail(e, "host pipeline: ordering after the caller's stream");
    // A call with another staging layout (workspace or slot size) than the
    // previous one waits until both slots of the previous one are free: its
    // slots need not coincide with the old ones.
    if (P->last_ws != workspace || P->last_slot != L.slot) {
        for (int s = 0; s < 2 && e == cudaSuccess; ++s) e = cudaStreamWaitEvent(P->h2d, P->freed[s], 0);
        if (e != cudaSuccess) return cuda_fail(e, "host pipeline: ordering after the previous staging");
        P->last_ws = workspace;
        P->last_slot = L.slot;
    }
    for (long long b0 = 0; b0 < B && rc == ATTN_OK; b0 += L.cb) {
        const long long nb = B - b0 < L.cb ? B - b0 : L.cb;
        const int slot = static_cast<int>(P->chunks & 1);
        ++P->chunks;
        char* base = static_cast<char*>(workspace) + slot * L.slot;
        e = cudaStreamWaitEvent(P->h2d, P->freed[slot], 0);
        for (int x = 0; x < L.n_in && e == cudaSuccess; ++x)
            e = cudaMemcpyAsync(base + L.in_off[x], static_cast<const char*>(in[x]) + b0 * L.in_seq[x],
                                nb * L.in_seq[x], cudaMemcpyHostToDevice, P->h2d);
        if (e == cudaSuccess) e = cudaEventRecord(P->loaded[slot], P->h2d);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(P->comp, P->loaded[slot], 0);
        if (e != cudaSuccess) {
            rc = cuda_fail(e, "host pipeline: host-to-device copy");
            break;
        }
        rc = compute(static_cast<int>(nb), base, P->comp);
        if (rc != ATTN_OK) break;
        e = cudaEventRecord(P->computed[slot], P->comp);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(P->d2h, P->computed[slot], 0);
        for (int x = 0; x < L.n_out && e == cudaSuccess; ++x)
            e = cudaMemcpyAsync(static_cast<char*>(out[x]) + b0 * L.out_seq[x], base + L.out_off[x],
                                nb * L.out_seq[x], cudaMemcpyDeviceToHost, P->d2h);
        if (e == cudaSuccess) e = cudaEventRecord(P->freed[slot], P->d2h);
        if (e != cudaSuccess) rc = cuda_fail(e, "host pipeline: device-to-host copy");
    }
    // The caller's stream resumes after everything queued above.
    e = cudaEventRecord(P->done, P->d2h);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(user, P->done, 0);
    if (e != cudaSuccess && rc == ATTN_OK) rc = cuda_fail(e, "host pipeline: ordering the caller's stream");
    return rc;
}

// Scratch of the FP8 host forward per sequence: Q8, K8, V8 codes and the
// three block-scale arrays.
void fp8_scratch(int H, int H_kv, int N, int d, size_t s[6]) {
    const size_t nblk = (static_cast<size_t>(N) + 127) / 128;
    s[0] = static_cast<size_t>(N) * H * d;
    s[1] = s[2] = static_cast<size_t>(N) * H_kv * d;
    s[3] = static_cast<size_t>(H) * nblk * 4;
    s[4] = s[5] = static_cast<size_t>(H_kv) * nblk * 4;
}

}  // namespace

extern "C" {

size_t attn_fwd_host_workspace_size(int B, int H, int H_kv, int N, int d) {
    Staging L;
    if (!fwd_staging(B, H, H_kv, N, d, nullptr, 0, &L)) return 0;
    return 2 * L.slot;
}

int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N,
                  int d, int causal, float scale, int window, void* workspace, size_t workspace_bytes,
                  void* stream) {
    g_err[0] = '\0';
    int rc = check_common(q, k, v, o, lse, B, H, N, d, window);
    if (rc != ATTN_OK) return rc;
    if (H_kv <= 0 || H % H_kv != 0)
        return fail(ATTN_ERR_INVALID_ARG, "key/value heads (%d) must divide query heads (%d)", H_kv, H);
    if (static_cast<long long>(B) * H * N == 0) return ATTN_OK;
    Staging L;
    fwd_staging(B, H, H_kv, N, d, nullptr, 0, &L);
    const void* in[3] = {q, k, v};
    void* out[2] = {o, lse};
    return host_pipeline(in, out, B, L, workspace, workspace_bytes, stream, "attn_fwd_host",
                         [&](int nb, char* base, cudaStream_t s) {
                             return launch_forward(false, base + L.in_off[0], base + L.in_off[1], base + L.in_off[2],
                                                   base + L.out_off[0], reinterpret_cast<float*>(base + L.out_off[1]),
                                                   nb, H, H_kv, N, d, causal, scale, window, nullptr, nullptr,
                                                   nullptr, s);
                         });
}

size_t attn_fwd_fp8_host_workspace_size(int B, int H, int H_kv, int N, int d) {
    Staging L;
    size_t sc[6];
    if (H <= 0 || H_kv <= 0 || N <= 0 || d <= 0) return 0;
    fp8_scratch(H, H_kv, N, d, sc);
    if (!fwd_staging(B, H, H_kv, N, d, sc, 6, &L)) return 0;
    return 2 * L.slot;
}

int attn_fwd_fp8_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv,
                      int N, int d, int causal, float scale, int window, int mode, unsigned long long sign_seed,
                      void* workspace, size_t workspace_bytes, void* stream) {
    g_err[0] = '\0';
    int rc = check_common(q, k, v, o, lse, B, H, N, d, window);
    if (rc != ATTN_OK) return rc;
    if (H_kv <= 0 || H % H_kv != 0)
        return fail(ATTN_ERR_INVALID_ARG, "key/value heads (%d) must divide query heads (%d)", H_kv, H);
    if (mode != 0 && mode != 1)
        return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_fp8_host: mode %d (0 or 1; the per-tensor mode spans chunks)",
                    mode);
    if (static_cast<long long>(B) * H * N == 0) return ATTN_OK;
    Staging L;
    size_t sc[6];
    fp8_scratch(H, H_kv, N, d, sc);
    fwd_staging(B, H, H_kv, N, d, sc, 6, &L);
    size_t soff[6];
    for (int x = 0; x < 6; ++x)
        soff[x] = x == 0 ? L.scratch_off : soff[x - 1] + up256(static_cast<size_t>(L.cb) * sc[x - 1]);
    const void* in[3] = {q, k, v};
    void* out[2] = {o, lse};
    return host_pipeline(in, out, B, L, workspace, workspace_bytes, stream, "attn_fwd_fp8_host",
                         [&](int nb, char* base, cudaStream_t s) {
                             float* qs = reinterpret_cast<float*>(base + soff[3]);
                             float* ks = reinterpret_cast<float*>(base + soff[4]);
                             float* vs = reinterpret_cast<float*>(base + soff[5]);
                             int r = attn_fp8_prep_qkv(base + L.in_off[0], base + L.in_off[1], base + L.in_off[2],
                                                       base + soff[0], base + soff[1], base + soff[2], qs, ks, vs, nb,
                                                       H, H_kv, N, d, mode, sign_seed, s);
                             if (r != ATTN_OK) return r;
                             return launch_forward(true, base + soff[0], base + soff[1], base + soff[2],
                                                   base + L.out_off[0], reinterpret_cast<float*>(base + L.out_off[1]),
                                                   nb, H, H_kv, N, d, causal, scale, window, qs, ks, vs, s);
                         });
}

}  // extern "C"

namespace {

// The backward's parts: Q, K, V, O, LSE, dO in; dQ, dK, dV out; the
// backward's own workspace for one chunk as scratch.
bool bwd_staging(int B, int H, int H_kv, int N, int d, Staging* L) {
    if (B <= 0 || H <= 0 || H_kv <= 0 || N <= 0 || d <= 0) return false;
    const size_t q_seq = static_cast<size_t>(N) * H * d * 2, kv_seq = static_cast<size_t>(N) * H_kv * d * 2;
    const size_t l_seq = static_cast<size_t>(H) * N * 4;
    const size_t in[6] = {q_seq, kv_seq, kv_seq, q_seq, l_seq, q_seq}, out[3] = {q_seq, kv_seq, kv_seq};
    if (!staging(B, in, 6, out, 3, nullptr, 0, L)) return false;
    // one chunk's backward workspace (not a per-sequence size: added whole)
    L->slot += up256(static_cast<size_t>(attn::bwd_workspace(static_cast<int>(L->cb), H, N, d).bytes));
    return true;
}

}  // namespace

extern "C" {

size_t attn_bwd_host_workspace_size(int B, int H, int H_kv, int N, int d) {
    Staging L;
    if (!bwd_staging(B, H, H_kv, N, d, &L)) return 0;
    return 2 * L.slot;
}

int attn_bwd_host(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                  void* dq, void* dk, void* dv, int B, int H, int H_kv, int N, int d, int causal, float scale,
                  int window, void* workspace, size_t workspace_bytes, void* stream) {
    g_err[0] = '\0';
    int rc = check_common(q, k, v, o, lse, B, H, N, d, window);
    if (rc != ATTN_OK) return rc;
    if (d != 128 && d != 64) return fail(ATTN_ERR_UNSUPPORTED, "attn_bwd_host supports head_dim 64 and 128 (got %d)", d);
    if (H_kv <= 0 || H % H_kv != 0)
        return fail(ATTN_ERR_INVALID_ARG, "key/value heads (%d) must divide query heads (%d)", H_kv, H);
    if (static_cast<long long>(B) * H * N == 0) return ATTN_OK;
    if (!dout || !dq || !dk || !dv) return fail(ATTN_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return fail(ATTN_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    Staging L;
    bwd_staging(B, H, H_kv, N, d, &L);
    const size_t bwd_ws = up256(static_cast<size_t>(attn::bwd_workspace(static_cast<int>(L.cb), H, N, d).bytes));
    const void* in[6] = {q, k, v, o, lse, dout};
    void* out[3] = {dq, dk, dv};
    return host_pipeline(in, out, B, L, workspace, workspace_bytes, stream, "attn_bwd_host",
                         [&](int nb, char* base, cudaStream_t s) {
                             return attn_bwd(base + L.in_off[0], base + L.in_off[1], base + L.in_off[2],
                                             base + L.in_off[3], reinterpret_cast<const float*>(base + L.in_off[4]),
                                             base + L.in_off[5], base + L.out_off[0], base + L.out_off[1],
                                             base + L.out_off[2], base + L.scratch_off, bwd_ws, nb, H, H_kv, N, d,
                                             causal, scale, window, s);
                         });
}

}  // extern "C"
