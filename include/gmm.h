/*
 * gmm.h — C ABI of the GB300 (sm_103a) MoE grouped matmul library.
 *
 * The operation (a grouped matrix multiply, "GMM"): the rows of an activation
 * matrix X[M,K] are sorted by expert into G contiguous groups of sizes
 * group_sizes[0..G); group g owns rows [off_g, off_g + n_g), off being the
 * exclusive prefix sum of the sizes, and is multiplied by its own expert
 * weight W[g][K,N] ("MoE 优化的探索", §3.7.2: a grouped GEMM is a set of
 * independent per-expert GEMMs scheduled in one kernel; "GEMM Kernel
 * 性能优化十问", Q6 for the shapes).  Output rows from S = sum(group_sizes) up
 * to M belong to no group and are written as zeros ("实现差距：GMM Kernel（V1
 * vs V2）", §3.6).
 *
 * Conventions shared by every call
 *   - Pointers are DEVICE pointers unless stated otherwise.  The caller owns
 *     every buffer (including the workspace); the library never allocates
 *     device memory.  Every device pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous: they validate their arguments on the
 *     host, enqueue kernels on `stream` and return.
 *   - Host-checked errors (null pointer, shape, alignment, workspace size)
 *     return immediately and launch nothing.
 *   - Data-dependent errors (a negative group size, sum(group_sizes) > M) and
 *     a kernel's bounded wait running out set a sticky error word inside the
 *     workspace; the kernels then stop early and the outputs are undefined.
 *     gmm_get_device_status() reads and clears that word.  No kernel traps.
 *     Every wait is limited to 2 s of GPU time by default; the environment
 *     variable GMM_WAIT_LIMIT_MS (a positive number of milliseconds, read
 *     once per process) changes the limit for every entry point.
 *   - On GMM_ERR_CUDA (and the host-side errors that name a cause),
 *     gmm_last_cuda_error() gives the calling thread's last message.
 *   - Row-major layouts; bf16 = IEEE bfloat16; e4m3 = OCP FP8 E4M3 (max 448).
 *   - K and N are multiples of 128 (the quantization block); 1 <= G <= 4096;
 *     0 <= M < 2^31.  M = 0, or every group empty, is valid.
 *   - The grouped calls first derive the group metadata (offsets, row tiles)
 *     from group_sizes into the workspace.  group_sizes = NULL skips that step
 *     and reuses the metadata already in the workspace: written by
 *     gmm_group_metadata or by an earlier grouped call with the same G and M,
 *     enqueued earlier on the same stream (the layers of one MoE block share
 *     their routing, so one metadata pass serves all their grouped calls).
 */
#ifndef GMM_GB300_H
#define GMM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GMM_OK = 0,
  GMM_ERR_NULL = 1,         /* a required pointer is NULL */
  GMM_ERR_SHAPE = 2,        /* a size is out of range or not a multiple of 128 */
  GMM_ERR_ALIGN = 3,        /* a pointer is not 16-byte aligned */
  GMM_ERR_UNSUPPORTED = 4,  /* no GPU of compute capability 10.3 is current */
  GMM_ERR_CUDA = 5,         /* a CUDA runtime / driver call failed */
  GMM_ERR_GROUP_SIZES = 6,  /* device-detected: negative size or sum > M */
  GMM_ERR_TIMEOUT = 7,      /* device-detected: a bounded wait ran out */
  GMM_ERR_WORKSPACE = 8     /* workspace NULL or smaller than gmm_workspace_bytes */
} gmm_status;

/* Human-readable name of a status code (static storage). */
const char* gmm_status_string(gmm_status status);

/* Message of the last CUDA error seen by this thread's calls (static storage). */
const char* gmm_last_cuda_error(void);

/*
 * Bytes of device workspace the grouped calls need for G groups and M rows:
 * a status word, the group offsets, the row-tile list and the groups ordered
 * by size.  The workspace must be zero-filled once before its first use (its
 * first word is the sticky error word); afterwards it may be reused by any number of calls issued on
 * one stream.  Two calls that run concurrently need two workspaces.
 */
size_t gmm_workspace_bytes(int G, int64_t M);

/*
 * a1 — group metadata.  ("MoE 优化的探索", §3.7.2: tiles carry their expert id
 * and are located through offsets; "实现差距：GMM Kernel（V1 vs V2）", §1/§2.2:
 * the metadata is filled on the device.)
 * Reads group_sizes int32[G] (device) and writes into `workspace`:
 *   int32 word[0]  sticky error bits (1: a negative size, 2: sum > M,
 *                  4: a bounded wait ran out), OR-ed, never cleared here
 *   int32 word[1]  1 if this call's sizes were valid, else 0
 *   int32 word[2]  S = sum(group_sizes)        (M when invalid)
 *   int32 word[3]  T = number of row tiles      (0 when invalid)
 *   int32 word[4], word[5]  set to 0: the work counters of tgmm_bf16 and of
 *                  the FP8 forward with one CTA per tile (units claimed, CTAs
 *                  finished); each such launch claims its units from them and
 *                  its last CTA sets them back to 0
 *   int32 word[6]  T2 = number of 256-row tiles (0 when invalid)
 *   int32 word[8 + g], g = 0..G  exclusive prefix sums off_g (off_G = S)
 *   int32x4 tiles[T] at byte offset gmm_tiles_offset(G): {g, row0, row1, 0},
 *                  every group cut into consecutive tiles of at most 128 rows,
 *                  groups in order, empty groups contributing none.
 *   int32 order[G] at byte offset gmm_tiles_offset(G) + 16 * (ceil(M/128) + G):
 *                  the group ids sorted by size, largest first (ties by id);
 *                  the tgmm kernels take their work largest groups first.
 *   int32x4 pair_tiles[T2] at byte offset (that of order) + 16 * ceil(G/4):
 *                  {g, row0, row1, 0} as above with tiles of at most 256
 *                  rows, the row tiles of the CTA-pair FP8 kernel.
 * The grouped calls below run this step themselves unless they are given
 * group_sizes = NULL, in which case they read what this call (or an earlier
 * grouped call) left in the workspace.
 */
gmm_status gmm_group_metadata(const int32_t* group_sizes, int G, int64_t M, void* workspace,
                              size_t workspace_bytes, void* stream);
size_t gmm_tiles_offset(int G);

/*
 * a2 — dynamic LHS quantization in 1x128 blocks ("GEMM Kernel 性能优化十问",
 * Q2: one scale per row per 128 elements; "实现差距：GMM Kernel（V1 vs V2）",
 * §3.3: absmax -> scale = absmax / 448 -> inv = (scale == 0 ? 0 : 1/scale)
 * -> q = e4m3(x * inv)).  Scale and product are IEEE fp32, rounding to
 * nearest; the e4m3 cast rounds to nearest even and saturates at 448.
 *   x   bf16 [M, K]
 *   xq  e4m3 [M, K]            (one byte per element)
 *   xs  fp32 [K/128, M]        (scale of row m, block kb at xs[kb*M + m])
 */
gmm_status gmm_quantize_lhs(const void* x, int64_t M, int64_t K, void* xq, float* xs, void* stream);

/*
 * a3 — offline RHS quantization in 128x128 blocks (Q2: weights are static,
 * one scale per 128x128 block, computed ahead of time), same per-block rule.
 *   w   bf16 [G, K, N]
 *   wq  e4m3 [G, N, K]   NOTE: transposed ("K-major"): wq[(g*N + n)*K + k]
 *                        holds the code of w[g][k][n]
 *   ws  fp32 [G, K/128, N/128]
 * For the fused gate/up weight pass N = 2 * N_out (gate columns first).
 */
gmm_status gmm_quantize_rhs(const void* w, int G, int64_t K, int64_t N, void* wq, float* ws, void* stream);

/*
 * a4-a6 — FP8 blockwise GMM forward ("GEMM Kernel 性能优化十问", Q1/Q3: the
 * K loop runs over many 128-wide quantization blocks; each block's exact
 * partial product is promoted into an fp32 accumulator with the LHS row scale
 * times the RHS block scale; "实现差距：GMM Kernel（V1 vs V2）", §3.3):
 *   out[m,n] = bf16( sum_kb P_kb[m,n] * xs[kb,m] * ws[g,kb,n/128] ),
 *   P_kb[m,n] = sum_{k in kb} xq[m,k] * wq[g,k,n]   (fp32 on the tensor core)
 * fuse_silu_mul = 1 (§3.5 of the V1/V2 page): wq holds 2N columns (gate
 * [0,N), up [N,2N)) and out[m,n] = bf16(silu(y_gate) * y_up), silu(v) =
 * v / (1 + exp(-v)), applied to the fp32 accumulators.
 *   xq, xs    as written by gmm_quantize_lhs (M rows, K columns)
 *   wq, ws    as written by gmm_quantize_rhs (G, K, N or 2N)
 *   out       bf16 [M, N]; rows >= S are written as zeros
 * GMM_ERR_SHAPE also when the work units, (ceil(M/128) + G) row tiles times
 * N/256 (or N/128) column blocks, reach 2^31 (far beyond any real layer).
 */
gmm_status gmm_fp8_fwd(const void* xq, const float* xs, const void* wq, const float* ws,
                       const int32_t* group_sizes, int G, int64_t M, int64_t K, int64_t N,
                       int fuse_silu_mul, void* out, void* workspace, size_t workspace_bytes,
                       void* stream);

/*
 * Tile configuration of the FP8 forward, the space the autotuner searches
 * ("GEMM Kernel 性能优化十问", Q8: tile sizes chosen by a search over measured
 * candidates, each checked for accuracy).  Every configuration computes the
 * same sums in the same order (each output element is one row tile's K loop
 * of one unit, every K block's partial promoted in K order); a field left 0
 * keeps the default.
 *   bn          columns of W per work unit: 128 or 256.  256 needs
 *               N % 256 == 0 or fuse_silu_mul = 1 (default then); 128 is not
 *               available with fuse_silu_mul = 1 or with cta_group = 2.
 *   ctas        persistent CTAs, 1 .. the number of SMs (default: one per SM,
 *               rounded down to even for cta_group = 2, which needs an even
 *               count)
 *   unit_order  1: row-tile major, the column blocks of a row tile run side
 *               by side (default); 2: column-block major, the row tiles that
 *               share a column block of an expert's weights run side by side
 *   cta_group   1: one CTA per 128-row tile, MMA M = 128, N = bn, two TMEM
 *               partial buffers (default); 2: CTA pairs on 256-row tiles (the
 *               MMA of two SMs, M = 256), each K block as two N = 128 halves
 *               into four TMEM buffers, the weight tile split between the
 *               pair (needs N % 256 == 0 or fuse_silu_mul = 1, bn 0 or 256
 *               and an even ctas)
 *   stages      slots of the shared-memory operand ring: cta_group 1 with
 *               bn 256: 2 or 3 (default 3); with bn 128: 3, 4 (default) or 5;
 *               cta_group 2: 3 to 5 (default 5) fused, 3 or 4 (default 4)
 *               otherwise
 *   tmem_bufs   TMEM partial buffers the MMA rotates through: 2 with bn 256,
 *               2 (default) or 4 with bn 128 (then all 512 TMEM columns), 4
 *               for cta_group 2
 * A value outside these returns GMM_ERR_UNSUPPORTED before any launch.
 */
typedef struct {
  int bn;
  int ctas;
  int unit_order;
  int cta_group;
  int stages;
  int tmem_bufs;
} gmm_fp8_tile_config;

/*
 * gmm_fp8_fwd with a tile configuration (config = NULL: the defaults, exactly
 * gmm_fp8_fwd).  Same arguments, layouts, results and errors otherwise.
 */
gmm_status gmm_fp8_fwd_tiled(const void* xq, const float* xs, const void* wq, const float* ws,
                             const int32_t* group_sizes, int G, int64_t M, int64_t K, int64_t N,
                             int fuse_silu_mul, void* out, void* workspace, size_t workspace_bytes, void* stream,
                             const gmm_fp8_tile_config* config);

/*
 * FP8 forward of the gate/up layer with the next layer's quantization fused
 * into its epilogue: "MoE 优化的探索" §5.1 names the step between Linear-1 and
 * Linear-2 "SwiGLU / FP8 Cast"; here the wi kernel emits, besides (optionally)
 * h = bf16(silu(gate) * up), its 1x128 e4m3 quantization directly:
 *   hq, hs  = exactly what gmm_quantize_lhs(h, M, N, hq, hs) would write
 *             (the absmax is taken over the bf16-rounded h; same fp32 arithmetic)
 * Arguments as gmm_fp8_fwd with fuse_silu_mul = 1 (wq holds 2N columns), plus
 *   h   bf16 [M, N] or NULL (then only hq, hs are written)
 *   hq  e4m3 [M, N];  hs  fp32 [N/128, M]; rows >= S get codes 0 and scale 0.
 */
gmm_status gmm_fp8_fwd_swiglu_quant(const void* xq, const float* xs, const void* wq, const float* ws,
                                    const int32_t* group_sizes, int G, int64_t M, int64_t K, int64_t N, void* h,
                                    void* hq, float* hs, void* workspace, size_t workspace_bytes, void* stream);

/*
 * gmm_fp8_fwd_swiglu_quant with a tile configuration (gmm_fp8_tile_config
 * above; bn must be 0 or 256, the fused units being 256 columns of W;
 * config = NULL: exactly gmm_fp8_fwd_swiglu_quant).
 */
gmm_status gmm_fp8_fwd_swiglu_quant_tiled(const void* xq, const float* xs, const void* wq, const float* ws,
                                          const int32_t* group_sizes, int G, int64_t M, int64_t K, int64_t N,
                                          void* h, void* hq, float* hs, void* workspace, size_t workspace_bytes,
                                          void* stream, const gmm_fp8_tile_config* config);

/*
 * Sub-byte weights ("实现差距：GMM Kernel（V1 vs V2）", §3.4: the V2 kernel
 * takes int4 / float4_e2m1fn weight tiles and keeps the blockwise fp32-scale
 * arithmetic; §4.1 lists MXFP4 weights as the missing piece).  Here: FP4 E2M1
 * weight codes (1 sign, 2 exponent bits with bias 1, 1 mantissa bit; values
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives) with one fp32 scale per
 * 128x128 block, scale = absmax / 6 (the same rule as gmm_quantize_rhs with
 * 6, the largest E2M1 value, in place of 448), codes = e2m1(w * (1/scale)),
 * nearest even, saturating at 6.  The weights stay packed (half the bytes of
 * e4m3) until the copy into shared memory expands them for the tensor core.
 *   w    bf16 [G, K, N]
 *   wq4  packed codes [G, N, K/2] bytes (K-major): byte (g*N + n)*K/2 + k/2
 *        holds the code of w[g][k][n] for even k in its low 4 bits and that
 *        of k + 1 in its high 4 bits; 32-byte aligned
 *   ws   fp32 [G, K/128, N/128]
 */
gmm_status gmm_quantize_rhs_w4(const void* w, int G, int64_t K, int64_t N, void* wq4, float* ws, void* stream);

/*
 * The FP8 forward (gmm_fp8_fwd_tiled, gmm_fp8_fwd_swiglu_quant_tiled) with
 * 4-bit weights: the activations are e4m3 in 1x128 blocks as before, the
 * weights E2M1 codes as written by gmm_quantize_rhs_w4 (wq4 32-byte aligned),
 * each 128-wide K block's partial P_kb = sum_k xq[m,k] * wq4[g,k,n] formed on
 * the tensor core (e4m3 x e2m1, fp32) and promoted with xs[kb,m] *
 * ws[g,kb,n/128] exactly as for e4m3 weights.  Same arguments, layouts,
 * tile configurations (config may be NULL) and errors otherwise.
 */
gmm_status gmm_fp8_w4_fwd(const void* xq, const float* xs, const void* wq4, const float* ws,
                          const int32_t* group_sizes, int G, int64_t M, int64_t K, int64_t N, int fuse_silu_mul,
                          void* out, void* workspace, size_t workspace_bytes, void* stream,
                          const gmm_fp8_tile_config* config);
gmm_status gmm_fp8_w4_fwd_swiglu_quant(const void* xq, const float* xs, const void* wq4, const float* ws,
                                       const int32_t* group_sizes, int G, int64_t M, int64_t K, int64_t N, void* h,
                                       void* hq, float* hs, void* workspace, size_t workspace_bytes, void* stream,
                                       const gmm_fp8_tile_config* config);

/*
 * a7 — bf16 GMM forward, unquantized (the BF16 baseline of "GEMM Kernel
 * 性能优化十问", Q7/Q10 step 4): out[m,n] = bf16(sum_k x[m,k] * w[g,k,n]),
 * fp32 accumulation; fuse_silu_mul as for gmm_fp8_fwd.
 *   x    bf16 [M, K]
 *   w    bf16 [G, K, N or 2N]   (natural layout, N contiguous)
 *   out  bf16 [M, N]; rows >= S are written as zeros
 */
gmm_status gmm_bf16_fwd(const void* x, const void* w, const int32_t* group_sizes, int G, int64_t M,
                        int64_t K, int64_t N, int fuse_silu_mul, void* out, void* workspace,
                        size_t workspace_bytes, void* stream);

/*
 * bf16 dgrad, the activation gradient of the expert GEMM: the "bwd" phase of
 * "GEMM Kernel 性能优化十问", Q4 (fwd, bwd and tgmm each get their own tiling),
 * kept in bf16 like the rest of the backward pass (Q5):
 *   dx[m,k] = bf16( sum_n dy[m,n] * w[g,k,n] ),  m in group g; fp32 accumulation
 *   dy  bf16 [M, N];  w  bf16 [G, K, N] (the forward weight, natural layout);
 *   dx  bf16 [M, K]; rows >= S are written as zeros.
 */
gmm_status gmm_bf16_dgrad(const void* dy, const void* w, const int32_t* group_sizes, int G, int64_t M,
                          int64_t K, int64_t N, void* dx, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * a8 — tgmm, the expert weight gradient ("GEMM Kernel 性能优化十问", Q4:
 * dW[K,N] += X^T[K,M] dY[M,N], M is the reduction; Q5: the backward pass
 * stays bf16, unquantized):
 *   dw[g][k,n] = bf16( sum_{m in group g} x[m,k] * dy[m,n] ), fp32 accumulation;
 *   dw[g] = 0 for an empty group.
 *   x   bf16 [M, K];  dy  bf16 [M, N];  dw  bf16 [G, K, N]
 * GMM_ERR_SHAPE also when G * (K/128) * (N/256, or N/128 when N % 256 != 0)
 * output tiles exceed 2^30.
 */
gmm_status tgmm_bf16(const void* x, const void* dy, const int32_t* group_sizes, int G, int64_t M,
                     int64_t K, int64_t N, void* dw, void* workspace, size_t workspace_bytes,
                     void* stream);

/*
 * Tile configuration of tgmm_bf16, the space the autotuner searches for it
 * ("GEMM Kernel 性能优化十问", Q4: the fwd, bwd and tgmm phases each get their
 * own tiling; Q8: chosen by a search over measured candidates).  The fields
 * apply to the CTA-pair kernel (K % 256 == 0); every configuration computes
 * the same sums in the same order.  A field left 0 keeps the default.
 *   stages       slots of its operand ring with 256-column units (N % 256 ==
 *                0): 4, 5 or 6 (default 6); 128-column units always use 8
 *   claim_ahead  units the pair's scheduler may hold beyond those its
 *                producer has started: 1..12 (default 3); independently of it
 *                the scheduler claims only while fewer than 8 chunks (64 rows
 *                each) are queued ahead of its producer
 *   max_batch    most units one claim takes once the units are small: 1..4
 *                (default 4).  The units are ordered largest group first; when
 *                the largest group has more than twice the chunks of the
 *                smallest, claims alternate between the two ends of that order
 * A value outside these returns GMM_ERR_UNSUPPORTED before any launch.
 */
typedef struct {
  int stages;
  int claim_ahead;
  int max_batch;
} gmm_tgmm_tile_config;

/* tgmm_bf16 with a tile configuration (config = NULL: exactly tgmm_bf16). */
gmm_status tgmm_bf16_tiled(const void* x, const void* dy, const int32_t* group_sizes, int G, int64_t M,
                           int64_t K, int64_t N, void* dw, void* workspace, size_t workspace_bytes,
                           void* stream, const gmm_tgmm_tile_config* config);

/*
 * gmm_fp8_fwd without a workspace argument, for callers that cannot allocate
 * device memory when they run the layer: code running under a framework whose
 * allocator owns all device memory, a runtime that must not allocate after
 * start-up (fixed budgets, real-time loops), or a plug-in that is only handed
 * its input and output buffers.  (The pages have no counterpart: this is an
 * interface choice of this library, not part of the method.)
 *
 * Same arguments, layouts and result as gmm_fp8_fwd, minus the workspace.
 * The group metadata goes to a 64 KiB array in the library's own device
 * memory (a file-scope __device__ variable, reserved on every GPU that loads
 * the library and held until the process exits).  The call allocates nothing:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 *   - Limit: gmm_workspace_bytes(G, M) must be <= 65536 (for example G <= 1024
 *     with M <= 65536, or G <= 256 with M <= 262144); larger sizes return
 *     GMM_ERR_WORKSPACE and launch
 *     nothing.
 *   - The first call on each device does a one-time set-up with that device
 *     current (it looks up the device address of the array with
 *     cudaGetSymbolAddress); make that first call before any stream capture.
 *   - Every call on a device shares the one array and leaves its contents for
 *     the next; each call rewrites all it reads.  Calls that overlap on the
 *     GPU (different streams without ordering between them) race on it and
 *     must not be issued.
 *   - Bounded waits, GMM_WAIT_LIMIT_MS and gmm_last_cuda_error() behave as
 *     for every other entry point.
 *   - Device-detected errors (invalid group_sizes, a wait that ran out) are
 *     not reported by this entry point: the array's error word is cleared at
 *     the start of every call and cannot be read through this ABI; on such an
 *     error the output is undefined.  Validate group_sizes beforehand, or use
 *     gmm_fp8_fwd with a workspace and gmm_get_device_status.
 */
gmm_status gmm_fp8_fwd_noalloc(const void* xq, const float* xs, const void* wq, const float* ws,
                               const int32_t* group_sizes, int G, int64_t M, int64_t K, int64_t N,
                               int fuse_silu_mul, void* out, void* stream);

/*
 * Diagnostic of the failure path (the pages have no counterpart: this checks
 * the library's own safety mechanism).  Launches one small kernel whose
 * threads wait, through the same bounded wait every kernel of this library
 * uses, on a barrier that nothing ever completes: after limit_ms (1..10000)
 * the wait gives up, the other waiting warps stop through the shared abort
 * word, GMM_ERR_TIMEOUT's bit is set in the workspace's sticky error word and
 * the kernel returns; gmm_get_device_status() then reports GMM_ERR_TIMEOUT.
 * The GPU context stays usable.  workspace: any zero-initialised workspace
 * (at least 16 bytes).
 */
gmm_status gmm_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int limit_ms, void* stream);

/*
 * Synchronizes `stream`, reads the workspace's sticky error word, clears it
 * and maps it to a status: GMM_ERR_TIMEOUT if a wait ran out, else
 * GMM_ERR_GROUP_SIZES if some call saw invalid group sizes, else GMM_OK.
 */
gmm_status gmm_get_device_status(void* workspace, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GMM_GB300_H */
