/*
 * attn.h -- C ABI of the GB300 (sm_103a) fused exact attention (forward,
 * FP8 prep, backward).
 *
 * What is computed (FlashAttention-3 deep-reading report, "第三层" intro and
 * §3.1-§3.3; "Efficient Attention & FlashAttention", "数学机理"):
 *
 *     O   = softmax(scale * Q K^T + mask) V          per (batch, head)
 *     LSE = log(sum_j exp(scale * q_i . k_j))        natural log, per row,
 *                                                    over the visible keys
 *
 * evaluated tile by tile with an online softmax (running row max m, running
 * row sum l, the O accumulator rescaled when m grows, one division by l at
 * the end) so that the N x N score matrix never reaches device memory.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Layout (the practitioner's FA3 re-test post, §4.2): Q, K, V and O are
 *    contiguous (batch B, seqlen N, heads H, head_dim d) tensors, d fastest;
 *    LSE is a contiguous (B, H, N) float32 tensor.
 *  - d must be 64, 128 or 256.  B, H, N >= 0; an empty problem is a no-op.
 *  - Mask: key j is visible to query i iff (causal == 0 || j <= i) and
 *    (window <= 0 || j > i - window).  With causal != 0 and window = W > 0
 *    each query sees the W most recent keys including itself (a sliding
 *    window).  Key tiles that no query of a query tile can see are skipped,
 *    not masked.
 *  - scale <= 0 or non-finite selects 1 / sqrt(d).
 *  - All pointers are DEVICE pointers, 16-byte aligned, owned by the
 *    caller; the library allocates no device memory per call and keeps no
 *    reference after the call returns.  Tensor memory (TMEM) is allocated and
 *    freed inside each kernel.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Argument errors are detected before any launch.
 *  - Return value: ATTN_OK or a negative attn_status.  The text of the last
 *    error of the calling thread is available from attn_last_error_string().
 *  - Under the causal and window masks alone every query sees at least
 *    itself.  Only attn_fwd_sparse can leave a row with no visible key (its
 *    block mask hides every key block of the row's query tile); such rows
 *    get O = 0 and LSE = -inf.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = -1,    /* bad pointer, size, alignment or mode      */
    ATTN_ERR_UNSUPPORTED = -2,    /* head_dim / device not supported           */
    ATTN_ERR_CUDA = -3,           /* a CUDA runtime / driver call failed       */
    ATTN_ERR_DEVICE_TIMEOUT = -4  /* a kernel gave up waiting (see below)      */
} attn_status;

/*
 * attn_fwd -- bf16 fused attention forward.
 *   q, k, v : const bf16 (B, N, H, d)
 *   o       : bf16 (B, N, H, d), written
 *   lse     : float32 (B, H, N), written
 * The exponentials, the running max/sum and the accumulators are float32;
 * P is rounded to bf16 for the P V product; the row sum l is accumulated
 * from the unrounded float32 probabilities.
 * Design (deep-reading report §3.1, §3.2): TMA-fed K/V shared-memory ring,
 * warp-specialised load / MMA / softmax roles, tcgen05 MMAs with the S and
 * O accumulators in tensor memory.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int H, int N, int d, int causal, float scale, int window,
             void* stream);

/*
 * attn_fwd_fp8 -- FP8 (e4m3) fused attention forward (deep-reading report
 * §2.2 and §3.3: block quantization and incoherent processing).
 *   q8, k8, v8          : const e4m3 (B, N, H, d) from attn_fp8_prep
 *   q_scale, k_scale,
 *   v_scale             : const float32 (B, H, ceil(N / 128)): the scale of
 *                         each 128-token block, so that the real value of an
 *                         element is scale * e4m3 value
 *   o                   : bf16 (B, N, H, d), written
 *   lse                 : float32 (B, H, N), written
 * Q and K must have been rotated with the same seed (or not at all); the
 * rotation leaves Q K^T unchanged.  V's block scale lies on the contraction
 * dimension of P V, so it is folded into P before P is rounded to e4m3:
 * P8 = e4m3(P * 16 * v_scale_j / vmax) with vmax the largest V block scale
 * of the (batch, head) and P <= 2^4.8 (the row maximum used in P moves only
 * when a score exceeds it by more than 4.8 in log2 units, so P * 16 <= 445.7
 * stays below e4m3's largest value, 448); O = (sum P8 V8) * vmax / (16 * l).  d must be 64, 128 or 256 (ATTN_ERR_UNSUPPORTED otherwise).
 */
int attn_fwd_fp8(const void* q8, const void* k8, const void* v8, void* o, float* lse,
                 int B, int H, int N, int d, int causal, float scale, int window,
                 const float* q_scale, const float* k_scale, const float* v_scale,
                 void* stream);

/*
 * attn_fwd_gqa / attn_fwd_fp8_gqa -- grouped-query and multi-query attention
 * (deep-reading report §3.4: FA3 keeps FA2's index adjustment for MQA/GQA,
 * so K and V are not duplicated in memory).  As attn_fwd / attn_fwd_fp8,
 * except that K and V (and, for FP8, k_scale and v_scale) have H_kv heads:
 *   k, v (k8, v8)       : (B, N, H_kv, d)
 *   k_scale, v_scale    : float32 (B, H_kv, ceil(N / 128))
 * H_kv must divide H; query head h reads key/value head h / (H / H_kv).
 * H_kv == H is multi-head attention (attn_fwd and attn_fwd_fp8 call these
 * with H_kv = H); H_kv == 1 is multi-query attention.
 */
int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int H_kv, int N, int d, int causal, float scale, int window,
                 void* stream);
int attn_fwd_fp8_gqa(const void* q8, const void* k8, const void* v8, void* o, float* lse,
                     int B, int H, int H_kv, int N, int d, int causal, float scale, int window,
                     const float* q_scale, const float* k_scale, const float* v_scale,
                     void* stream);

/*
 * attn_fp8_prep -- fused rotation + block quantisation of one tensor
 * (deep-reading report §2.2 / §3.3).
 *   x      : const bf16 (B, N, H, d)
 *   x8     : e4m3 (B, N, H, d), written
 *   scales : float32 (B, H, ceil(N / block_rows)), written
 *   block_rows : tokens per scale block; must be 128
 *   mode   : 0 = per-block scales;
 *            1 = per-block scales after incoherent processing
 *                r = x D H_d / sqrt(d)  (D = diag(+-1) from sign_seed,
 *                H_d the Sylvester Hadamard matrix); skipped when is_v != 0;
 *            2 = one scale for the whole tensor (the per-tensor baseline),
 *                stored in every entry of `scales`.
 *   sign_seed : seed of the +-1 diagonal: sign c is -1 iff bit 63 of
 *            splitmix64 output c (state = sign_seed) is set.
 *   is_v   : nonzero for V (never rotated).
 * scale = amax / 448 of the block (1 for an all-zero block); each element is
 * r / scale rounded to nearest-even e4m3 and saturated to +-448.  amax, the
 * scale and the division are float32.  For modes 0 and 1 at d = 64 and 128
 * the product x (D H) is taken on the tensor cores (D H is a +-1 matrix,
 * exact in bf16; fp32 accumulation), so r may differ from a float32
 * butterfly evaluation in its last bits.
 */
int attn_fp8_prep(const void* x, void* x8, float* scales, int B, int H, int N, int d,
                  int block_rows, int mode, unsigned long long sign_seed, int is_v,
                  void* stream);

/*
 * attn_fp8_prep_qkv -- attn_fp8_prep of Q, K and V of one attention call in
 * one launch (deep-reading report §2.2 / §3.3): Q and K rotated in mode 1
 * (the same sign_seed, so Q K^T is unchanged), V never rotated.
 *   q          : const bf16 (B, N, H, d);  k, v : const bf16 (B, N, H_kv, d)
 *   q8, k8, v8 : e4m3, the same shapes, written
 *   q_scale    : float32 (B, H, ceil(N / 128)); k_scale, v_scale : (B, H_kv,
 *                ceil(N / 128)); written
 *   mode, sign_seed : as attn_fp8_prep (block_rows is 128).
 * H_kv must divide H.  Modes 0 and 1 at d = 64 and 128 run as one launch
 * over the blocks of all three tensors; d = 256 and mode 2 run as three
 * attn_fp8_prep calls.  Results are those of three attn_fp8_prep calls.
 * Errors: ATTN_ERR_INVALID_ARG / ATTN_ERR_UNSUPPORTED as attn_fp8_prep,
 * before any launch.
 */
int attn_fp8_prep_qkv(const void* q, const void* k, const void* v, void* q8, void* k8, void* v8,
                      float* q_scale, float* k_scale, float* v_scale, int B, int H, int H_kv,
                      int N, int d, int mode, unsigned long long sign_seed, void* stream);

/*
 * attn_fp8_prep_rope -- rotary position embedding fused with the FP8 prep of
 * Q or K (deep-reading report §2.2 / §3.3: the block quantisation costs
 * nothing extra when it rides inside the memory-bound rotary-embedding
 * pass).  As attn_fp8_prep with is_v = 0, except that each row of token n is
 * first turned by RoPE (Su et al., "RoFormer", 2021):
 *     a' = a cos(n, i) - b sin(n, i),   b' = a sin(n, i) + b cos(n, i)
 * for pair index i < d/2, with the pair (a, b) = elements (i, i + d/2) when
 * interleaved == 0 ("half-split") or (2i, 2i + 1) when interleaved != 0.
 * The products and sums are float32, each rounded (no fused multiply-add).
 * Then, in this order, the Hadamard rotation (mode 1) and the quantiser.
 *   rope_cos, rope_sin : const float32 (N, d/2), device, 16-byte aligned,
 *                        owned by the caller; row n serves token n of every
 *                        batch and head.
 * Errors: as attn_fp8_prep; a NULL or unaligned table is
 * ATTN_ERR_INVALID_ARG.
 */
int attn_fp8_prep_rope(const void* x, void* x8, float* scales, const float* rope_cos,
                       const float* rope_sin, int B, int H, int N, int d, int block_rows,
                       int mode, unsigned long long sign_seed, int interleaved, void* stream);

/*
 * attn_fwd_sparse -- bf16 forward with a block-sparse key mask (the
 * practitioner's FA3 post, §3.3 and §4.3: the caller marks which KV blocks a
 * Q block skips; the decision is per (Q block, KV block), not per element).
 * As attn_fwd_gqa, except that
 *   block_mask : const uint8 (B, H, T, T), device, T = ceil(N / 128), owned
 *                by the caller; entry [b][h][i][j] != 0 lets query rows
 *                [128 i, 128 i + 128) of (b, h) see key rows [128 j,
 *                128 j + 128).  It is ANDed with the causal and window masks.
 * Key blocks a query block does not see are skipped, not computed.  A row
 * that sees no key gets O = 0 and LSE = -inf.  d must be 64, 128 or 256.
 * Errors: as attn_fwd_gqa; a NULL block_mask is ATTN_ERR_INVALID_ARG.
 */
int attn_fwd_sparse(const void* q, const void* k, const void* v, void* o, float* lse,
                    const unsigned char* block_mask, int B, int H, int H_kv, int N, int d,
                    int causal, float scale, int window, void* stream);

/*
 * attn_fwd_host_workspace_size / attn_fwd_host -- attn_fwd_gqa on HOST
 * buffers.  The pages' forward reads Q, K, V from and writes O, LSE to device
 * memory; this entry is the same computation for a caller whose tensors live
 * in host memory (no counterpart in the pages).  The batch is cut into
 * chunks of whole sequences; for each chunk the library copies Q, K, V to
 * one of two device staging slots, runs the forward on it and copies O and
 * LSE back, with the copies of one chunk overlapping the forward and the
 * copies of its neighbours (three library-owned streams, created once per
 * device; events order them).  Consecutive calls overlap the same way.
 *   q, k, v, o, lse : HOST pointers with the layouts of attn_fwd_gqa
 *                     (16-byte aligned; page-locked memory, e.g. from
 *                     cudaHostAlloc, is what lets the copies overlap)
 *   workspace       : device, at least attn_fwd_host_workspace_size(B, H,
 *                     H_kv, N, d) bytes, 256-byte aligned, owned by the
 *                     caller (the two staging slots)
 *   B, H, H_kv, N, d, causal, scale, window : as attn_fwd_gqa
 * The call is asynchronous on `stream`: its copies start after the work
 * already queued on `stream`, and work queued on `stream` afterwards starts
 * after O and LSE are in host memory, so the caller synchronizes `stream`
 * before reading them and keeps the buffers alive until then.  Calls may
 * share a workspace, on any streams: the library orders the reuse of its
 * staging slots (two calls in flight on two streams overlap the copies of
 * one with those of the other).  Errors: as attn_fwd_gqa;
 * a NULL, unaligned or too small workspace is ATTN_ERR_INVALID_ARG;
 * ATTN_ERR_CUDA if a copy or a launch fails part-way (the chunks queued
 * before it still complete in order on `stream`).
 * attn_fwd_host_workspace_size returns 0 for invalid sizes.
 */
size_t attn_fwd_host_workspace_size(int B, int H, int H_kv, int N, int d);
int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                  int H_kv, int N, int d, int causal, float scale, int window, void* workspace,
                  size_t workspace_bytes, void* stream);

/*
 * attn_fwd_fp8_host_workspace_size / attn_fwd_fp8_host -- the FP8 path on
 * HOST buffers: per chunk of sequences, the bf16 Q, K, V copied in are
 * prepared (attn_fp8_prep with `mode` and `sign_seed`: Q and K rotated in mode
 * 1, V never) and fed to attn_fwd_fp8_gqa, and O, LSE are copied back, staged
 * and overlapped exactly as attn_fwd_host (no counterpart in the pages).
 *   q, k, v         : HOST bf16 (B, N, H / H_kv, d), as attn_fwd_host
 *   o, lse          : HOST outputs, as attn_fwd_host
 *   mode            : 0 (per-block scales) or 1 (per-block scales after the
 *                     rotation); the per-tensor mode 2 is refused
 *                     (ATTN_ERR_INVALID_ARG) since its one scale would span
 *                     chunks
 *   workspace       : device, at least attn_fwd_fp8_host_workspace_size(B, H,
 *                     H_kv, N, d) bytes, 256-byte aligned (the two slots also
 *                     hold the e4m3 codes and block scales of their chunk)
 * d must be 64, 128 or 256.  Ordering, sharing and errors as attn_fwd_host.
 */
size_t attn_fwd_fp8_host_workspace_size(int B, int H, int H_kv, int N, int d);
int attn_fwd_fp8_host(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int H_kv, int N, int d, int causal, float scale, int window, int mode,
                      unsigned long long sign_seed, void* workspace, size_t workspace_bytes,
                      void* stream);

/*
 * attn_bwd_workspace_size / attn_bwd -- backward of attn_fwd / attn_fwd_gqa
 * (deep-reading report §3.4: FA3 keeps FA2's recompute strategy; five
 * matrix products against the forward's two).  For a loss L with upstream
 * gradient dout = dL/dO:
 *     P_ij = exp(scale q_i . k_j - LSE_i),  dP_ij = dout_i . v_j,
 *     D_i = dout_i . o_i,  dS_ij = P_ij (dP_ij - D_i),
 *     dq_i = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i,
 *     dv_j = sum_i P_ij dout_i
 * (sums over visible pairs; dk, dv of a key/value head sum over the query
 * heads of its group).
 *   q, dout, o          : const bf16 (B, N, H, d), device; o and lse are the
 *                         forward's outputs for the same q, k, v and mask
 *   k, v                : const bf16 (B, N, H_kv, d)
 *   lse                 : const float32 (B, H, N) from the forward
 *   dq                  : bf16 (B, N, H, d), written
 *   dk, dv              : bf16 (B, N, H_kv, d), written
 *   workspace           : device, at least attn_bwd_workspace_size(B, H, N, d)
 *                         bytes, 256-byte aligned, owned by the caller; its
 *                         contents are scratch (overwritten by every call,
 *                         so calls sharing one workspace must be ordered on
 *                         one stream)
 *   B, H, H_kv, N, d, causal, scale, window : as attn_fwd_gqa
 * d must be 64 or 128 (ATTN_ERR_UNSUPPORTED otherwise).  Three
 * launches on `stream`: D and the zeroed float32 dQ accumulator, the fused
 * backward, and the conversion of dQ to bf16.  Errors: as attn_fwd_gqa; a
 * NULL, unaligned or too small workspace is ATTN_ERR_INVALID_ARG.
 * attn_bwd_workspace_size returns 0 for negative sizes.
 */
size_t attn_bwd_workspace_size(int B, int H, int N, int d);
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, void* workspace,
             size_t workspace_bytes, int B, int H, int H_kv, int N, int d, int causal,
             float scale, int window, void* stream);

/*
 * attn_bwd_host_workspace_size / attn_bwd_host -- attn_bwd on HOST buffers
 * (no counterpart in the pages): per chunk of whole sequences, q, k, v, o,
 * lse and dout are copied to a device staging slot, the backward runs there
 * (its scratch is part of the slot) and dq, dk, dv are copied back, staged
 * and overlapped exactly as attn_fwd_host.
 *   q, k, v, o, lse, dout : HOST inputs with the layouts of attn_bwd
 *   dq, dk, dv            : HOST outputs, written
 *   workspace             : device, at least attn_bwd_host_workspace_size(B,
 *                           H, H_kv, N, d) bytes, 256-byte aligned
 * d must be 64 or 128.  Ordering, sharing and errors as attn_fwd_host.
 */
size_t attn_bwd_host_workspace_size(int B, int H, int H_kv, int N, int d);
int attn_bwd_host(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, int B, int H, int H_kv, int N,
                  int d, int causal, float scale, int window, void* workspace,
                  size_t workspace_bytes, void* stream);

/*
 * attn_bwd_noalloc / attn_bwd_noalloc_max_scratch -- attn_bwd for callers
 * that cannot allocate device memory: code running where cudaMalloc is not
 * allowed or not wanted (inside a framework's own allocator or memory pool,
 * in a process whose memory budget is fixed up front, or in a library layer
 * that must not own device buffers).  There is no counterpart in the paper;
 * this is a convenience of this library.
 * Arguments as attn_bwd, without the workspace: the scratch (about
 * 4 * B * H * ceil(N / 128) * 128 * (d + 2) bytes, attn_bwd_workspace_size)
 * lives in one static device buffer of attn_bwd_noalloc_max_scratch() bytes
 * (256 MiB), created on every GPU that loads this library's device code and
 * held until the process exits.  A larger problem is rejected with
 * ATTN_ERR_INVALID_ARG and a message naming the sizes; attn_bwd with a
 * caller workspace has no such limit.
 *  - The first call on a device looks up the buffer's device address (one
 *    cudaGetSymbolAddress); make that first call before any stream capture.
 *  - Every call on a device shares the one buffer: calls whose kernels can
 *    overlap on the GPU (different streams without ordering) race and give
 *    wrong gradients.  Order them on one stream.  Each call rewrites the
 *    parts it reads first (the dQ accumulator is zeroed), so sequential
 *    calls are independent.
 *  - Nothing is allocated: no cudaMalloc, cudaFree or allocating library
 *    call.
 */
size_t attn_bwd_noalloc_max_scratch(void);
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dout, void* dq, void* dk, void* dv, int B, int H, int H_kv,
                     int N, int d, int causal, float scale, int window, void* stream);

/*
 * attn_device_status -- waits for `stream`, then reads and clears the
 * library's device status word.  Every wait inside the kernels is bounded;
 * a kernel that gives up records the site in this word and returns instead
 * of hanging.  Returns ATTN_OK, ATTN_ERR_DEVICE_TIMEOUT (*site, if not NULL,
 * receives the site code) or ATTN_ERR_CUDA.
 */
int attn_device_status(void* stream, int* site);

/*
 * attn_set_wait_limit -- cycles (SM clock) a kernel waits on one barrier
 * before giving up; 0 restores the default (about two seconds).  Applies to
 * launches made after the call, from any thread.
 */
int attn_set_wait_limit(unsigned long long cycles);

/*
 * attn_fwd_work_order -- the order in which a causal forward at head_dim
 * 128 without grouped heads (H_kv = H, no block mask) hands its work items
 * to the grid; host code only, no GPU needed (inspection and testing).  A
 * work item is one batch*head and one query block of 256 rows.  The grid
 * takes the items in rounds of `grid`: round m goes to the CTAs in order
 * when m is even and in reverse when odd.  The order: the n mod grid
 * lightest items (query block ascending, then head) form the last, partial
 * round; the others, taken head by head (query block descending within a
 * head), are cut into rounds of `grid`, each numbered heaviest query block
 * first, then by head.
 *   n_mblocks : query blocks per head, ceil(N / 256)
 *   BH        : B * H
 *   grid      : CTAs of the launch, min(n_mblocks * BH, SM count)
 *   out       : HOST array of `capacity` entries; entry i = query block of
 *               item i | (its batch*head) << 16
 * Returns the number of entries written (n_mblocks * BH), or 0 when such a
 * launch uses the closed-form order instead (more than 2048 items), when
 * `capacity` is too small, or for invalid sizes.
 */
int attn_fwd_work_order(int n_mblocks, int BH, int grid, unsigned int* out, int capacity);

/* Text of the last error of the calling thread ("" if none). */
const char* attn_last_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
