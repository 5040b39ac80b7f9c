// fp64 CPU oracle for the fused exact-attention forward and its FP8 prep.
//
// TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
// benchmark's CPU-baseline leg load this library.  It shares no code, header
// or constant table with the CUDA path, and the CUDA path never calls it.
//
// Sources (the pages the method is described on):
//  [R] "深度解读报告：FlashAttention-3（2024）" (FlashAttention-3 deep-reading
//      report): §3 intro (tiling with running max m and running sum l, the
//      N x N matrix never written to HBM), §2.2 and §3.3 (block quantization,
//      incoherent processing M = diag(+-1) x Hadamard with M M^T = I),
//      §4.3 (errors are measured against an FP64 reference implementation).
//  [E] "Efficient Attention & FlashAttention: 解释 FlashAttention-2/3 的改进",
//      "数学机理" (FA2 normalises once per query block; the result is still
//      the plain softmax attention).
//
// What is computed.  The tiled, online-softmax method reaches exactly (up to
// rounding order) the plain definition of attention, so the oracle is that
// definition, written out in double precision with every score of a row
// materialised and a two-pass softmax:
//     s_j   = scale * sum_c q_ic k_jc           for every visible key j
//     m     = max_j s_j
//     l     = sum_j exp(s_j - m)
//     O_i   = sum_j exp(s_j - m) v_j / l
//     LSE_i = m + log(l)                        (natural log)
// Visibility of key j to query i: j <= i when causal; j > i - window when
// window > 0; and, with a block-sparse mask (the practitioner's FA3 post,
// §3.3: the caller decides per query block and key block whether the pair
// takes part), mask[b][h][i / 128][j / 128] != 0.  A row that sees no key
// gets O = 0 and LSE = -inf.
//
// FP8 prep (block quantization + incoherent processing, [R] §2.2 / §3.3):
//     r   = x M  with M = D H_d / sqrt(d)   (Q and K; V is not rotated)
//     per block of `block_rows` consecutive tokens of one (batch, head):
//         amax  = max |r|           scale = amax / 448  (1 when amax == 0)
//         code  = e4m3(r / scale)   (round to nearest even, saturate to 448)
// The rotation is a dense d x d product in double.  The quantisation decision
// (amax, scale, r / scale and the rounding to e4m3) is taken in binary32,
// the precision the CUDA path takes it in, so that a code is comparable bit
// for bit.  The OCP 8-bit floating point specification (OFP8, E4M3: 1 sign,
// 4 exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 is
// NaN, largest finite 448) defines the encoder below.
//
// Backward ([R] §3.4 appendix note: FA3 keeps FA2's recompute strategy,
// five matrix products against the forward's two).  With L a scalar loss
// and dO = dL/dO given, the gradients of the same definition are
//     P_ij  = exp(s_ij - LSE_i)                 (0 for invisible keys)
//     dP_ij = dO_i . v_j
//     D_i   = sum_j P_ij dP_ij                  (softmax Jacobian term)
//     dS_ij = P_ij (dP_ij - D_i)
//     dQ_i  = scale sum_j dS_ij k_j
//     dK_j  = scale sum_(h in group) sum_i dS_ij q_i
//     dV_j  = sum_(h in group) sum_i P_ij dO_i
// computed in double in two passes: per query row (LSE, D, dQ), then per
// key row (dK, dV) with P and dS recomputed from the stored LSE and D.
//
// Rotary position embedding before the quantiser (the report's §2.2 and
// §3.3: the block quantisation can ride inside the memory-bound rotary
// embedding kernel).  RoPE itself is the rotation of Su et al., "RoFormer:
// Enhanced Transformer with Rotary Position Embedding" (2021): the pair
// (a, b) of token n and pair index i turns by the angle of table entry
// (n, i):  a' = a cos - b sin,  b' = a sin + b cos.  Pairs are (i, i + d/2)
// ("half-split") or (2i, 2i + 1) ("interleaved").  The caller supplies the
// binary32 cos / sin tables, shape (N, d/2).  The rotation is evaluated in
// binary32 with each product and each sum rounded (no fused multiply-add),
// the precision the CUDA path computes it in, because its result feeds the
// quantisation decision.  Order on Q and K: RoPE, then the Hadamard rotation,
// then the quantiser (x R_n M: M acts on the already position-rotated row,
// and (q R_m M)(k R_n M)^T = (q R_m)(k R_n)^T).
//
// Random signs of D: bit 63 of successive outputs of splitmix64 seeded with
// the caller's seed (Steele, Lea and Flood 2014; Vigna's public reference
// splitmix64.c): output c (c = 0, 1, ...) is mix(seed + (c + 1) * gamma).
// A set bit gives -1.
//
// Portable C++17; no intrinsics, runs the same on x86-64 and aarch64.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

double bf16_value(uint16_t bits) {
    uint32_t u = static_cast<uint32_t>(bits) << 16;
    float f;
    std::memcpy(&f, &u, sizeof f);
    return static_cast<double>(f);
}

bool key_visible_plain(long i, long j, int causal, int window) {
    if (causal && j > i) return false;
    if (window > 0 && j <= i - window) return false;
    return true;
}

int pick_threads(int requested, long work_items) {
    int t = requested > 0 ? requested : static_cast<int>(std::thread::hardware_concurrency());
    if (t < 1) t = 1;
    if (work_items < t) t = static_cast<int>(std::max<long>(1, work_items));
    return t;
}

template <class F>
void parallel_for(long count, int nthreads, F&& body) {
    int t = pick_threads(nthreads, count);
    if (t == 1) {
        for (long i = 0; i < count; ++i) body(i);
        return;
    }
    std::atomic<long> next{0};
    std::vector<std::thread> pool;
    pool.reserve(t);
    for (int w = 0; w < t; ++w) {
        pool.emplace_back([&] {
            for (long i = next.fetch_add(1); i < count; i = next.fetch_add(1)) body(i);
        });
    }
    for (auto& th : pool) th.join();
}

// One query row of one (batch, head): the plain two-pass definition.
// in(b, n, h, c) reads element c of token n, head h of batch b from a
// (B, N, H, d) tensor.  probs (optional) receives the N softmax weights.
// plane: the (b, h) plane of a block mask, T x T with T = ceil(N / 128), or
// nullptr for none.
template <class In>
void attention_row(const In& qin, const In& kin, const In& vin, long b, long h, long i,
                   long N, long d, int causal, double scale, int window,
                   double* o_row, double* lse_out, double* probs, const uint8_t* plane = nullptr) {
    const long T = (N + 127) / 128;
    auto key_visible = [&](long ii, long j, int c, int w) {
        return key_visible_plain(ii, j, c, w) && (!plane || plane[(ii / 128) * T + j / 128] != 0);
    };
    std::vector<double> s(N, -std::numeric_limits<double>::infinity());
    std::vector<double> q(d);
    for (long c = 0; c < d; ++c) q[c] = qin(b, i, h, c);
    double m = -std::numeric_limits<double>::infinity();
    bool any = false;
    for (long j = 0; j < N; ++j) {
        if (!key_visible(i, j, causal, window)) continue;
        double acc = 0.0;
        for (long c = 0; c < d; ++c) acc += q[c] * kin(b, j, h, c);
        s[j] = scale * acc;
        if (!any || s[j] > m) m = s[j];
        any = true;
    }
    for (long c = 0; c < d; ++c) o_row[c] = 0.0;
    if (!any) {
        *lse_out = -std::numeric_limits<double>::infinity();
        if (probs) for (long j = 0; j < N; ++j) probs[j] = 0.0;
        return;
    }
    double l = 0.0;
    for (long j = 0; j < N; ++j) {
        if (!key_visible(i, j, causal, window)) { s[j] = 0.0; continue; }
        s[j] = std::exp(s[j] - m);
        l += s[j];
    }
    for (long j = 0; j < N; ++j) {
        if (!key_visible(i, j, causal, window)) continue;
        const double w = s[j];
        for (long c = 0; c < d; ++c) o_row[c] += w * vin(b, j, h, c);
    }
    for (long c = 0; c < d; ++c) o_row[c] /= l;
    *lse_out = m + std::log(l);
    if (probs) {
        for (long j = 0; j < N; ++j) probs[j] = key_visible(i, j, causal, window) ? s[j] / l : 0.0;
    }
}

// A (B, N, heads, d) tensor read by query head h: with grouped-query
// attention (deep-reading report §3.4) query head h reads key/value head
// h / group, where group = query heads / key-value heads.
struct Bf16Tensor {
    const uint16_t* p; long N, H, d, group;
    double operator()(long b, long n, long h, long c) const {
        return bf16_value(p[((b * N + n) * H + h / group) * d + c]);
    }
};
struct F64Tensor {
    const double* p; long N, H, d, group;
    double operator()(long b, long n, long h, long c) const { return p[((b * N + n) * H + h / group) * d + c]; }
};

// Output layout: o is (B, H, R, d) and lse is (B, H, R), R = number of rows
// computed (all N rows when rows == nullptr).
template <class In>
int run_attention(const In& q, const In& k, const In& v, double* o, double* lse,
                  int B, int H, int N, int d, int causal, double scale, int window,
                  const int* rows, int nrows, int nthreads, const uint8_t* block_mask = nullptr) {
    if (B < 0 || H < 0 || N < 0 || d <= 0) return -1;
    const long R = rows ? nrows : N;
    for (long r = 0; rows && r < R; ++r) if (rows[r] < 0 || rows[r] >= N) return -1;
    const long items = static_cast<long>(B) * H * R;
    parallel_for(items, nthreads, [&](long it) {
        const long r = it % R;
        const long bh = it / R;
        const long b = bh / H, h = bh % H;
        const long i = rows ? rows[r] : r;
        const long T = (static_cast<long>(N) + 127) / 128;
        const uint8_t* plane = block_mask ? block_mask + (b * H + h) * T * T : nullptr;
        attention_row(q, k, v, b, h, i, N, d, causal, scale, window,
                      o + it * d, lse + it, nullptr, plane);
    });
    return 0;
}

// ---- OCP FP8 E4M3 --------------------------------------------------------

double e4m3_decode_one(uint8_t code) {
    const int sign = code >> 7;
    const int e = (code >> 3) & 0xF;
    const int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return std::numeric_limits<double>::quiet_NaN();
    if (e == 0) v = std::ldexp(static_cast<double>(m), -9);          // m/8 * 2^-6
    else v = std::ldexp(8.0 + m, e - 7 - 3);                          // (1 + m/8) * 2^(e-7)
    return sign ? -v : v;
}

// Round half to even of a non-negative double that holds at most 53 bits.
double round_half_even(double x) {
    double f = std::floor(x);
    double r = x - f;
    if (r > 0.5) return f + 1.0;
    if (r < 0.5) return f;
    return (std::fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

// Encode with round-to-nearest-even and saturation to the largest finite
// magnitude (448); NaN encodes as 0x7F with the sign bit of the input.
uint8_t e4m3_encode_one(double x) {
    const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
    if (std::isnan(x)) return static_cast<uint8_t>(sign | 0x7F);
    double a = std::fabs(x);
    if (a >= 448.0) return static_cast<uint8_t>(sign | 0x7E);
    const double min_normal = std::ldexp(1.0, -6);
    if (a < min_normal) {
        // Subnormal grid: multiples of 2^-9 (exact scaling by a power of two).
        double n = round_half_even(std::ldexp(a, 9));
        if (n >= 8.0) return static_cast<uint8_t>(sign | (1 << 3));  // rounds up to 2^-6
        return static_cast<uint8_t>(sign | static_cast<int>(n));
    }
    int e2;
    std::frexp(a, &e2);            // a = f * 2^e2, f in [0.5, 1)
    int e = e2 - 1;                // a in [2^e, 2^(e+1))
    double n = round_half_even(std::ldexp(a, 3 - e));  // 8 <= n <= 16
    if (n >= 16.0) { n = 8.0; e += 1; }
    double val = std::ldexp(n, e - 3);
    if (val > 448.0) return static_cast<uint8_t>(sign | 0x7E);
    const int ef = e + 7;
    const int mf = static_cast<int>(n) - 8;
    return static_cast<uint8_t>(sign | (ef << 3) | mf);
}

// ---- splitmix64 signs and the Hadamard rotation --------------------------

uint64_t splitmix64_output(uint64_t seed, uint64_t c) {
    uint64_t z = seed + (c + 1) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

double sign_of(uint64_t seed, long c) { return (splitmix64_output(seed, c) >> 63) ? -1.0 : 1.0; }

// Sylvester ordering: H[r][c] = (-1)^popcount(r & c).
double sylvester(long r, long c) {
    unsigned long x = static_cast<unsigned long>(r & c);
    int parity = 0;
    while (x) { parity ^= 1; x &= x - 1; }
    return parity ? -1.0 : 1.0;
}

bool is_pow2(long d) { return d > 0 && (d & (d - 1)) == 0; }

// Backward pass 1, one query row i of query head h: LSE_i, D_i and dQ_i.
template <class In>
void backward_row(const In& qin, const In& kin, const In& vin, const In& doin, long b, long h, long i,
                  long N, long d, int causal, double scale, int window, double* dq_row, double* lse_out,
                  double* D_out) {
    std::vector<double> p(N), o(d);
    double lse;
    attention_row(qin, kin, vin, b, h, i, N, d, causal, scale, window, o.data(), &lse, p.data());
    std::vector<double> dout(d), dp(N, 0.0);
    for (long c = 0; c < d; ++c) dout[c] = doin(b, i, h, c);
    double D = 0.0;
    for (long j = 0; j < N; ++j) {
        if (!key_visible_plain(i, j, causal, window)) continue;
        double acc = 0.0;
        for (long c = 0; c < d; ++c) acc += dout[c] * vin(b, j, h, c);
        dp[j] = acc;
        D += p[j] * acc;
    }
    for (long c = 0; c < d; ++c) dq_row[c] = 0.0;
    for (long j = 0; j < N; ++j) {
        if (!key_visible_plain(i, j, causal, window)) continue;
        const double ds = p[j] * (dp[j] - D);
        for (long c = 0; c < d; ++c) dq_row[c] += ds * kin(b, j, h, c);
    }
    for (long c = 0; c < d; ++c) dq_row[c] *= scale;
    *lse_out = lse;
    *D_out = D;
}

// Backward pass 2, one key row j of key/value head hk: dK_j and dV_j summed
// over the query heads of the group and all query rows.
template <class In>
void backward_key(const In& qin, const In& kin, const In& vin, const In& doin, const double* lse,
                  const double* Dv, long b, long hk, long j, long N, long H, long d, long group, int causal,
                  double scale, int window, double* dk_row, double* dv_row) {
    for (long c = 0; c < d; ++c) dk_row[c] = dv_row[c] = 0.0;
    for (long h = hk * group; h < (hk + 1) * group; ++h) {
        const double* lse_h = lse + (b * H + h) * N;
        const double* D_h = Dv + (b * H + h) * N;
        for (long i = 0; i < N; ++i) {
            if (!key_visible_plain(i, j, causal, window)) continue;
            double s = 0.0, dp = 0.0;
            for (long c = 0; c < d; ++c) {
                s += qin(b, i, h, c) * kin(b, j, h, c);
                dp += doin(b, i, h, c) * vin(b, j, h, c);
            }
            const double P = std::exp(scale * s - lse_h[i]);
            const double ds = P * (dp - D_h[i]);
            for (long c = 0; c < d; ++c) {
                dk_row[c] += scale * ds * qin(b, i, h, c);
                dv_row[c] += P * doin(b, i, h, c);
            }
        }
    }
}

// q, dout, dq: (B, N, H, d); k, v, dk, dv: (B, N, Hkv, d).
template <class In>
int run_backward(const In& q, const In& k, const In& v, const In& dout, double* dq, double* dk, double* dv,
                 int B, int H, int Hkv, int N, int d, int causal, double scale, int window, int nthreads) {
    if (B < 0 || H < 0 || N < 0 || d <= 0 || Hkv <= 0 || H % Hkv != 0) return -1;
    const long group = H / Hkv;
    std::vector<double> lse(static_cast<size_t>(B) * H * N), Dv(static_cast<size_t>(B) * H * N);
    parallel_for(static_cast<long>(B) * H * N, nthreads, [&](long it) {
        const long i = it % N, bh = it / N, b = bh / H, h = bh % H;
        backward_row(q, k, v, dout, b, h, i, N, d, causal, scale, window, dq + ((b * N + i) * H + h) * d,
                     &lse[it], &Dv[it]);
    });
    parallel_for(static_cast<long>(B) * Hkv * N, nthreads, [&](long it) {
        const long j = it % N, bhk = it / N, b = bhk / Hkv, hk = bhk % Hkv;
        const long off = ((b * N + j) * Hkv + hk) * d;
        backward_key(q, k, v, dout, lse.data(), Dv.data(), b, hk, j, N, H, d, group, causal, scale, window,
                     dk + off, dv + off);
    });
    return 0;
}

}  // namespace

extern "C" {

int oracle_attn_bwd_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout,
                         double* dq, double* dk, double* dv, int B, int H, int Hkv, int N, int d, int causal,
                         double scale, int window, int nthreads) {
    if (Hkv <= 0 || H % Hkv != 0) return -1;
    const long g = H / Hkv;
    return run_backward(Bf16Tensor{q, N, H, d, 1}, Bf16Tensor{k, N, Hkv, d, g}, Bf16Tensor{v, N, Hkv, d, g},
                        Bf16Tensor{dout, N, H, d, 1}, dq, dk, dv, B, H, Hkv, N, d, causal, scale, window, nthreads);
}

int oracle_attn_bwd_f64(const double* q, const double* k, const double* v, const double* dout, double* dq,
                        double* dk, double* dv, int B, int H, int Hkv, int N, int d, int causal, double scale,
                        int window, int nthreads) {
    if (Hkv <= 0 || H % Hkv != 0) return -1;
    const long g = H / Hkv;
    return run_backward(F64Tensor{q, N, H, d, 1}, F64Tensor{k, N, Hkv, d, g}, F64Tensor{v, N, Hkv, d, g},
                        F64Tensor{dout, N, H, d, 1}, dq, dk, dv, B, H, Hkv, N, d, causal, scale, window, nthreads);
}

// Q has H heads, K and V have Hkv heads (Hkv divides H).
int oracle_attn_fwd_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         double* o, double* lse, int B, int H, int Hkv, int N, int d,
                         int causal, double scale, int window,
                         const int* rows, int nrows, int nthreads) {
    if (Hkv <= 0 || H % Hkv != 0) return -1;
    Bf16Tensor Q{q, N, H, d, 1}, K{k, N, Hkv, d, H / Hkv}, V{v, N, Hkv, d, H / Hkv};
    return run_attention(Q, K, V, o, lse, B, H, N, d, causal, scale, window, rows, nrows, nthreads);
}

// As oracle_attn_fwd_bf16 with a block mask (B, H, T, T), T = ceil(N / 128).
int oracle_attn_fwd_bf16_masked(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                double* o, double* lse, int B, int H, int Hkv, int N, int d,
                                int causal, double scale, int window, const uint8_t* block_mask,
                                const int* rows, int nrows, int nthreads) {
    if (Hkv <= 0 || H % Hkv != 0) return -1;
    Bf16Tensor Q{q, N, H, d, 1}, K{k, N, Hkv, d, H / Hkv}, V{v, N, Hkv, d, H / Hkv};
    return run_attention(Q, K, V, o, lse, B, H, N, d, causal, scale, window, rows, nrows, nthreads, block_mask);
}

int oracle_attn_fwd_f64_masked(const double* q, const double* k, const double* v,
                               double* o, double* lse, int B, int H, int Hkv, int N, int d,
                               int causal, double scale, int window, const uint8_t* block_mask,
                               const int* rows, int nrows, int nthreads) {
    if (Hkv <= 0 || H % Hkv != 0) return -1;
    F64Tensor Q{q, N, H, d, 1}, K{k, N, Hkv, d, H / Hkv}, V{v, N, Hkv, d, H / Hkv};
    return run_attention(Q, K, V, o, lse, B, H, N, d, causal, scale, window, rows, nrows, nthreads, block_mask);
}

int oracle_attn_fwd_f64(const double* q, const double* k, const double* v,
                        double* o, double* lse, int B, int H, int Hkv, int N, int d,
                        int causal, double scale, int window,
                        const int* rows, int nrows, int nthreads) {
    if (Hkv <= 0 || H % Hkv != 0) return -1;
    F64Tensor Q{q, N, H, d, 1}, K{k, N, Hkv, d, H / Hkv}, V{v, N, Hkv, d, H / Hkv};
    return run_attention(Q, K, V, o, lse, B, H, N, d, causal, scale, window, rows, nrows, nthreads);
}

// Softmax weights of one query row (length N; zero for hidden keys).
int oracle_attn_row_probs_f64(const double* q, const double* k, const double* v,
                              int B, int H, int N, int d, int causal, double scale, int window,
                              int b, int h, int i, double* probs) {
    if (b < 0 || b >= B || h < 0 || h >= H || i < 0 || i >= N) return -1;
    F64Tensor Q{q, N, H, d, 1}, K{k, N, H, d, 1}, V{v, N, H, d, 1};
    std::vector<double> orow(d);
    double lse;
    attention_row(Q, K, V, b, h, i, N, d, causal, scale, window, orow.data(), &lse, probs);
    return 0;
}

void oracle_e4m3_encode_f64(const double* x, uint8_t* out, long n) {
    for (long i = 0; i < n; ++i) out[i] = e4m3_encode_one(x[i]);
}

void oracle_e4m3_decode(const uint8_t* codes, double* out, long n) {
    for (long i = 0; i < n; ++i) out[i] = e4m3_decode_one(codes[i]);
}

// M = D H_d / sqrt(d), row-major d x d.
int oracle_rotation_matrix(int d, unsigned long long seed, double* M) {
    if (!is_pow2(d)) return -1;
    const double inv = 1.0 / std::sqrt(static_cast<double>(d));
    for (long r = 0; r < d; ++r) {
        const double sr = sign_of(seed, r);
        for (long c = 0; c < d; ++c) M[r * d + c] = sr * sylvester(r, c) * inv;
    }
    return 0;
}

void oracle_signs(int d, unsigned long long seed, double* out) {
    for (long c = 0; c < d; ++c) out[c] = sign_of(seed, c);
}

// RoPE of one row of token n (binary32 in, binary32 out, in place).
static void rope_row(float* r, long n, int d, const float* cos_t, const float* sin_t, int interleaved) {
    const long half = d / 2;
    for (long i = 0; i < half; ++i) {
        const long ia = interleaved ? 2 * i : i;
        const long ib = interleaved ? 2 * i + 1 : i + half;
        const float c = cos_t[n * half + i], s = sin_t[n * half + i];
        const float a = r[ia], b = r[ib];
        const float ac = a * c, bs = b * s, as = a * s, bc = b * c;   // each rounded
        r[ia] = ac - bs;
        r[ib] = as + bc;
    }
}

// x: bf16 (B, N, H, d) -> out: binary32 RoPE(x), same layout.
int oracle_rope_bf16(const uint16_t* x, float* out, const float* cos_t, const float* sin_t,
                     int B, int N, int H, int d, int interleaved, int nthreads) {
    if (B < 0 || N < 0 || H < 0 || d <= 0 || (d & 1)) return -1;
    parallel_for(static_cast<long>(B) * N * H, nthreads, [&](long row) {
        const long n = (row / H) % N;
        float* r = out + row * d;
        for (long c = 0; c < d; ++c) r[c] = static_cast<float>(bf16_value(x[row * d + c]));
        rope_row(r, n, d, cos_t, sin_t, interleaved);
    });
    return 0;
}

// x: bf16 (B, N, H, d).  x8: e4m3 codes (B, N, H, d).  scales: float
// (B, H, ceil(N / block_rows)).  rope_cos / rope_sin: optional binary32
// tables (N, d/2); when given, RoPE is applied first (Q and K only).  rotated (optional): the binary32 values r
// that were quantised, (B, N, H, d).
// mode 0: per-block scales; 1: per-block scales after the rotation (not for
// V); 2: one scale for the whole tensor (written to every block entry).
int oracle_fp8_quantize_rope(const uint16_t* x, uint8_t* x8, float* scales, float* rotated,
                             const float* rope_cos, const float* rope_sin, int rope_interleaved,
                             int B, int H, int N, int d, int block_rows, int mode,
                             unsigned long long seed, int is_v, int nthreads) {
    if (B < 0 || H < 0 || N < 0 || d <= 0 || block_rows <= 0 || mode < 0 || mode > 2) return -1;
    const bool rope = rope_cos != nullptr;
    if (rope && (is_v || (d & 1) || rope_sin == nullptr)) return -1;
    const bool rotate = (mode == 1) && !is_v;
    if (rotate && !is_pow2(d)) return -1;
    const long nblk = (N + block_rows - 1) / block_rows;
    const long total = static_cast<long>(B) * N * H * d;
    std::vector<float> r(total);
    std::vector<double> M;
    if (rotate) {
        M.resize(static_cast<size_t>(d) * d);
        oracle_rotation_matrix(d, seed, M.data());
    }
    // u = RoPE(x) (binary32) or u = x;  r = u M (double sum, rounded once to
    // binary32) or r = u.
    parallel_for(static_cast<long>(B) * N * H, nthreads, [&](long row) {
        const uint16_t* xr = x + row * d;
        float* rr = r.data() + row * d;
        std::vector<float> u(d);
        for (long c = 0; c < d; ++c) u[c] = static_cast<float>(bf16_value(xr[c]));
        if (rope) rope_row(u.data(), (row / H) % N, d, rope_cos, rope_sin, rope_interleaved);
        if (!rotate) {
            for (long c = 0; c < d; ++c) rr[c] = u[c];
            return;
        }
        for (long c = 0; c < d; ++c) {
            double acc = 0.0;
            for (long t = 0; t < d; ++t) acc += static_cast<double>(u[t]) * M[t * d + c];
            rr[c] = static_cast<float>(acc);
        }
    });
    auto at = [&](long b, long n, long h, long c) -> float& {
        return r[((b * N + n) * H + h) * d + c];
    };
    // Block amax (binary32 magnitudes; the maximum is exact).
    std::vector<float> amax(static_cast<size_t>(B) * H * nblk, 0.0f);
    parallel_for(static_cast<long>(B) * H * nblk, nthreads, [&](long it) {
        const long blk = it % nblk, bh = it / nblk, b = bh / H, h = bh % H;
        float a = 0.0f;
        for (long n = blk * block_rows; n < std::min<long>(N, (blk + 1) * block_rows); ++n)
            for (long c = 0; c < d; ++c) a = std::max(a, std::fabs(at(b, n, h, c)));
        amax[it] = a;
    });
    if (mode == 2) {
        float a = 0.0f;
        for (float v : amax) a = std::max(a, v);
        std::fill(amax.begin(), amax.end(), a);
    }
    for (size_t i = 0; i < amax.size(); ++i) {
        const float a = amax[i];
        scales[i] = (a > 0.0f) ? a / 448.0f : 1.0f;      // binary32 division
    }
    parallel_for(static_cast<long>(B) * N * H, nthreads, [&](long row) {
        const long h = row % H, bn = row / H, n = bn % N, b = bn / N;
        const float s = scales[(b * H + h) * nblk + n / block_rows];
        for (long c = 0; c < d; ++c) {
            const float y = r[row * d + c] / s;              // binary32 division
            x8[row * d + c] = e4m3_encode_one(static_cast<double>(y));
        }
    });
    if (rotated) std::memcpy(rotated, r.data(), sizeof(float) * total);
    return 0;
}

int oracle_fp8_quantize(const uint16_t* x, uint8_t* x8, float* scales, float* rotated,
                        int B, int H, int N, int d, int block_rows, int mode,
                        unsigned long long seed, int is_v, int nthreads) {
    return oracle_fp8_quantize_rope(x, x8, scales, rotated, nullptr, nullptr, 0, B, H, N, d, block_rows,
                                    mode, seed, is_v, nthreads);
}

}  // extern "C"
