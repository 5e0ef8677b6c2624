/*
 * dora.h -- C ABI of libdora: the DoRA weight-norm and compose hot path on
 * GB300 (sm_103a).
 *
 * Method source (cited below as "P1 ¶<opening words>"):
 *   P1 = web page "人工智能训练新突破：Anthropic团队破解大模型微调内存瓶颈难题"
 *        (techwalker.com, 2026-04-01), summarising arXiv:2603.22276.
 *
 * Notation: W0[out,in] frozen base weight, A[r,in] and B[out,r] the low-rank
 * adapter, s its scale, m[out] the DoRA magnitude; activations base = x W0^T
 * and lora = x A^T B^T (NOT pre-scaled by s) are [T,out].
 *
 *   n_i  = || W0_i + s (B A)_i ||                       (per output row)
 *   g_i  = m_i / n_i
 *   y    = base + (g-1)*base + g*s*lora                 (g broadcast over T)
 *   d_base = g*dy,  d_lora = s*g*dy,
 *   d_mag_j = sum_t dy[t,j] * (base[t,j] + s*lora[t,j]) / n_j   (n held constant)
 *
 * Conventions shared by every entry point:
 *   - Every data pointer is a DEVICE pointer owned by the caller.  The library
 *     never allocates, frees or synchronises; every call is asynchronous on
 *     `stream` (NULL = the legacy default stream).
 *   - Arrays are dense and row-major with the shapes given; no aliasing
 *     between any input and any output.
 *   - Argument errors are detected on the host before anything is launched and
 *     return a status with no side effect.  A failed launch returns
 *     DORA_ERR_CUDA.  Kernels that wait on on-chip barriers give up after a
 *     bounded time and record it in a device word read by dora_device_error().
 *   - Results are bitwise reproducible for a given shape on a given device.
 *   - Only sm_103 devices are accepted (DORA_ERR_ARCH otherwise).
 *   - The calls may be captured in a CUDA graph once the same call (same
 *     shapes and buffers) has run outside capture: the first call of a
 *     device sets up kernel attributes, and the first with a shape or a set
 *     of buffers builds the plan and tensor maps it then reuses.  A replay
 *     gives the same bits as the calls launched one by one.
 */
#ifndef DORA_H
#define DORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *dora_stream_t;

typedef enum {
  DORA_OK = 0,
  DORA_ERR_NULL = 1,       /* a required pointer is NULL                          */
  DORA_ERR_SHAPE = 2,      /* a size is negative, zero where not allowed, or too large */
  DORA_ERR_ALIGN = 3,      /* a pointer or row stride breaks an alignment rule    */
  DORA_ERR_DTYPE = 4,      /* unknown activation dtype                            */
  DORA_ERR_WORKSPACE = 5,  /* workspace NULL, misaligned or smaller than required */
  DORA_ERR_ARCH = 6,       /* current device is not sm_103                        */
  DORA_ERR_CUDA = 7,       /* a CUDA runtime/driver call or launch failed         */
  DORA_ERR_DEVICE = 8      /* a kernel's bounded on-chip wait gave up (see dora_device_error) */
} dora_status;

typedef enum {
  DORA_F32 = 0,            /* activations and their gradients are float32  */
  DORA_BF16 = 1            /* activations and their gradients are bfloat16 */
} dora_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char *dora_status_str(dora_status st);

/* ------------------------------------------------------------------------ */
/* (a) factored per-output-row weight norm                                   */
/* ------------------------------------------------------------------------ */

/*
 * Bytes of device workspace dora_norm_factored needs for this shape.  Pure
 * host arithmetic (no CUDA call); an upper bound valid on any device.  It grows
 * as O((out + in)*r + r^2) -- rank-dependent factors only, never out*in
 * (P1 ¶第一个创新是"因式分解规范化"技术: memory O(out*in) -> O(out*r + r^2)).
 * Returns 0 for an invalid shape.
 */
size_t dora_norm_factored_workspace(int64_t out, int64_t in, int64_t r);

/*
 * norm[i] = || W0_i + s (B A)_i ||,  g[i] = m[i] / norm[i]   for i < out.
 *
 * P1 ¶第一个创新是"因式分解规范化"技术: the squared norm is evaluated as a base
 * term, a cross term and a Gram term,
 *     n_i^2 = ||W0_i||^2 + 2 s <U_i, B_i> + s^2 B_i G B_i^T,
 *     U = W0 A^T [out,r],  G = A A^T [r,r],
 * so the out x in adapted weight is never formed.  The contractions run on the
 * tensor cores with every fp32 operand split as x = h + l (h = bf16(x),
 * l = bf16(x - h)): each product as three bf16 products h*h + l*h + h*l with
 * fp32 accumulation (dropped terms <= 3 * 2^-18 of the product); n^2 is
 * clamped at 0 before the square root; g is an IEEE division with no epsilon
 * (n = 0 gives inf/NaN).  Two launches (the split of A, then one cooperative
 * launch with one CTA per SM whose CTAs wait on one another through counters
 * in the workspace); a device that cannot hold every CTA at once gets
 * DORA_ERR_CUDA.  Plans and encoded tensor maps are cached per shape and per
 * buffer set, so repeated calls cost a few microseconds of host time.
 *
 *   W0    float32 [out, in]    16-byte aligned, in % 4 == 0
 *   A     float32 [r, in]      16-byte aligned
 *   B     float32 [out, r]     16-byte aligned (any r >= 1)
 *   m     float32 [out]        4-byte aligned
 *   s     adapter scale (e.g. alpha/sqrt(r))
 *   norm  float32 [out]  out
 *   g     float32 [out]  out
 *   workspace  >= dora_norm_factored_workspace(out,in,r) bytes, 256-byte
 *              aligned, caller-owned scratch; contents on entry are ignored
 *   Sizes: out >= 0 (0 is a no-op), in >= 1, r >= 1, r <= 1024,
 *          out, in < 2^31.
 */
dora_status dora_norm_factored(const float *W0, const float *A, const float *B,
                               const float *m, float s,
                               int64_t out, int64_t in, int64_t r,
                               float *norm, float *g,
                               void *workspace, size_t workspace_bytes,
                               dora_stream_t stream);

/* ------------------------------------------------------------------------ */
/* (a') the same norm for bf16 weights                                       */
/* ------------------------------------------------------------------------ */

/*
 * n0sq[i] = sum_j W0[i,j]^2 for a bfloat16 W0 [rows, cols], fp32 result in a
 * fixed summation order.  W0 is frozen during fine-tuning, so its row norms
 * are computed once and passed to every dora_norm_factored_bf16 call (the
 * base term of P1 ¶第一个创新是"因式分解规范化"技术).
 *   W0    bfloat16 [rows, cols]  16-byte aligned, cols % 8 == 0
 *   n0sq  float32 [rows]         4-byte aligned
 *   Sizes: rows >= 0 (0 is a no-op), cols >= 1, both < 2^31.
 */
dora_status dora_row_sumsq_bf16(const void *W0, int64_t rows, int64_t cols, float *n0sq,
                                dora_stream_t stream);

/* Bytes of workspace dora_norm_factored_bf16 needs (host arithmetic; 0 for an
 * invalid shape).  O(out + (out + r) r) bytes: s/2 G in three bf16 pieces,
 * partial sums, and B padded to a 16-byte row when r % 8 != 0. */
size_t dora_norm_factored_bf16_workspace(int64_t out, int64_t in, int64_t r);

/*
 * The factored norm of dora_norm_factored for bfloat16 W0, A and B (the same
 * definition, P1 ¶第一个创新是"因式分解规范化"技术), with the base term taken from
 * n0sq:
 *     n_i^2 = n0sq[i] + 2 s <U_i, B_i> + s^2 B_i G B_i^T,   g_i = m_i / n_i.
 * Products of bf16 values are exact in fp32, so U = W0 A^T and G = A A^T are
 * single bf16 tensor-core products with fp32 accumulation; s/2 G enters as three
 * bf16 pieces whose sum carries it to fp32 precision.  No adapter or weight is
 * converted or copied (B only when r % 8 != 0).
 *
 *   W0    bfloat16 [out, in]   16-byte aligned, in % 8 == 0
 *   A     bfloat16 [r, in]     16-byte aligned
 *   B     bfloat16 [out, r]    16-byte aligned (any r >= 1)
 *   m     float32 [out]        4-byte aligned
 *   n0sq  float32 [out]        ||W0_i||^2 (dora_row_sumsq_bf16), 4-byte aligned
 *   s, norm, g, workspace, sizes: as dora_norm_factored (workspace from
 *   dora_norm_factored_bf16_workspace).
 */
dora_status dora_norm_factored_bf16(const void *W0, const void *A, const void *B,
                                    const float *m, const float *n0sq, float s,
                                    int64_t out, int64_t in, int64_t r,
                                    float *norm, float *g,
                                    void *workspace, size_t workspace_bytes,
                                    dora_stream_t stream);

/* ------------------------------------------------------------------------ */
/* (a'') gradient through the norm (the variant with the norm not detached)  */
/* ------------------------------------------------------------------------ */

/* Bytes of workspace dora_norm_factored_bwd needs (host arithmetic; 0 for an
 * invalid shape).  O((out + in) r + r^2) bytes, never out*in. */
size_t dora_norm_factored_bwd_workspace(int64_t out, int64_t in, int64_t r);

/*
 * The part of dL/dA and dL/dB that flows through the row norm n, for a loss
 * that sees n only through g = m / n.  P1 is silent on a gradient through the
 * norm (its backward holds n constant, which is what dora_compose_bwd does);
 * this entry point is the plain chain rule for callers that do not detach it.
 * With d_mag = dL/dm as dora_compose_bwd writes it, dL/dn_i = -g_i d_mag_i and,
 * for V = W0 + s B A and c_i = (dL/dn_i) / n_i,
 *
 *   dB = s c (.) (W0 A^T + s B G),         G = A A^T
 *   dA = s (c (.) B)^T W0 + s^2 H A,       H = B^T diag(c) B
 *
 * evaluated in factored form (the out x in matrix V is never formed) on the
 * tensor cores with the same bf16 three-product split (x = h + l, each
 * product h h + l h + h l, fp32 accumulation) as dora_norm_factored.
 * The outputs are ONLY the norm's share: the caller adds the gradients of its
 * own lora = x A^T B^T product.  dA and dB are overwritten.
 *
 *   W0, A, B   float32, as for dora_norm_factored (16-byte aligned, in % 4 == 0)
 *   norm, g    float32 [out]  the forward's outputs (dora_norm_factored)
 *   d_mag      float32 [out]  dL/dm (dora_compose_bwd)
 *   dA         float32 [r, in]   dB  float32 [out, r]   (4-byte aligned)
 *   workspace  >= dora_norm_factored_bwd_workspace(out, in, r) bytes, 256-byte aligned
 *   Sizes as dora_norm_factored; out == 0 writes zeros to dA (an empty sum).
 * Launches at most 11 kernels (A split, B padding when r % 4 != 0, the split of
 * s c (.) B transposed, two Gram passes and their reductions, the dB and dA
 * passes and the fixed-order sums of their stream-K parts); results are
 * bitwise reproducible.
 */
dora_status dora_norm_factored_bwd(const float *W0, const float *A, const float *B,
                                   const float *norm, const float *g, const float *d_mag,
                                   float s, int64_t out, int64_t in, int64_t r,
                                   float *dA, float *dB,
                                   void *workspace, size_t workspace_bytes,
                                   dora_stream_t stream);

/* ------------------------------------------------------------------------ */
/* (b) fused compose, forward                                                */
/* ------------------------------------------------------------------------ */

/*
 * y = base + (g-1)*base + g*s*lora, one pass over [T,out].
 *
 * P1 ¶第二个创新是"融合Triton内核"技术 (four elementwise kernels fused into one)
 * and ¶从技术架构角度来看 / ¶他们在一个Qwen2-VL-7B适配器上的测量 (stable form with
 * the correction (g-1) kept explicit, fp32 intermediates).  Every element is
 * computed in fp32 and rounded once (nearest even) to the activation dtype.
 *
 *   act   DORA_F32 or DORA_BF16: dtype of base, lora and y
 *   base, lora  [T, out] of `act`
 *   g     float32 [out]
 *   y     [T, out] of `act`
 *   Sizes: T >= 0, out >= 0 (either 0 is a no-op).  Any out and any element
 *   alignment are accepted; the 128-bit path is taken when out is a multiple
 *   of 16/sizeof(act) and base, lora and y are 16-byte aligned.
 */
dora_status dora_compose_fwd(dora_dtype act, const void *base, const void *lora,
                             const float *g, float s, int64_t T, int64_t out,
                             void *y, dora_stream_t stream);

/* ------------------------------------------------------------------------ */
/* (b) fused compose, backward                                               */
/* ------------------------------------------------------------------------ */

/*
 * Bytes of device workspace dora_compose_bwd needs (fp32 partial column sums
 * of d_mag).  Pure host arithmetic; an upper bound valid on any device.
 */
size_t dora_compose_bwd_workspace(int64_t T, int64_t out);

/*
 * d_base = g*dy,  d_lora = s*g*dy,
 * d_mag[j] = (sum_t dy[t,j]*(base[t,j] + s*lora[t,j])) / norm[j].
 *
 * P1 ¶研究团队还设计了一个智能的三层调度系统 (fused backward in training) and
 * ¶研究团队还进行了广泛的收敛等价性验证 (d_mag reduction order).  The row norm is
 * treated as a constant (no gradient into A or B).  d_base and d_lora are
 * rounded once to `act`; d_mag is float32, summed in a fixed order (per-thread
 * token runs, then a fixed-order sum of the per-run partials), so it is
 * bitwise reproducible.  d_mag is overwritten, not accumulated.
 *
 *   act        dtype of grad_out, base, lora, d_base, d_lora
 *   grad_out, base, lora   [T, out] of `act`
 *   g, norm    float32 [out]
 *   d_base, d_lora  [T, out] of `act`
 *   d_mag      float32 [out]
 *   workspace  >= dora_compose_bwd_workspace(T,out) bytes, 256-byte aligned
 *   Sizes: T >= 0, out >= 0 (out == 0 is a no-op; T == 0 gives d_mag = 0).
 */
dora_status dora_compose_bwd(dora_dtype act, const void *grad_out, const void *base,
                             const void *lora, const float *g, const float *norm,
                             float s, int64_t T, int64_t out,
                             void *d_base, void *d_lora, float *d_mag,
                             void *workspace, size_t workspace_bytes,
                             dora_stream_t stream);

/* ------------------------------------------------------------------------ */
/* (b') compose backward without a workspace                                 */
/* ------------------------------------------------------------------------ */

/* Size, in floats, of the library's fixed device scratch array (4 MiB). */
#define DORA_NOALLOC_SCRATCH_FLOATS (1 << 20)

/*
 * Same results as dora_compose_bwd, but allocation-free for the caller: no
 * workspace argument.  The paper has no counterpart to this entry point; it
 * exists for callers that cannot allocate device memory where they run the
 * backward -- code embedded in an application that owns a fixed device memory
 * pool and exposes no allocator, or services that forbid cudaMalloc after
 * start-up because it synchronises the device and fragments shared memory.
 *
 * The d_mag partial sums go to one file-scope device array of
 * DORA_NOALLOC_SCRATCH_FLOATS floats, held on every GPU that loads the library
 * until the process exits.  The first call on a device looks up that array's
 * device address (cudaGetSymbolAddress, with the device current); make that
 * first call before any stream capture.  A device reset (cudaDeviceReset)
 * gives the device a new context and invalidates the address: the next call
 * looks it up again, so after a reset, too, make one call before any capture.
 * Every partial sum the call reads is
 * written earlier in the same call, so nothing needs clearing between calls,
 * but all calls share the one array: calls that overlap on the GPU (different
 * streams, or concurrent host threads on one device) race and give wrong
 * d_mag.  The call itself allocates nothing (no cudaMalloc/cudaFree, no
 * allocating library routine).
 *
 * Arguments, layouts and errors as dora_compose_bwd, plus: out must not exceed
 * DORA_NOALLOC_SCRATCH_FLOATS (DORA_ERR_SHAPE otherwise).  The call launches
 * exactly the grid dora_compose_bwd launches, so d_mag is bitwise the same.
 * That grid's partial rows times out stay below 4096 x the SM count floats,
 * which fits the array on any device with up to 256 SMs (GB300 has 152); a
 * device where it would not fit gets DORA_ERR_SHAPE before any launch.
 */
dora_status dora_compose_bwd_noalloc(dora_dtype act, const void *grad_out, const void *base,
                                     const void *lora, const float *g, const float *norm,
                                     float s, int64_t T, int64_t out,
                                     void *d_base, void *d_lora, float *d_mag,
                                     dora_stream_t stream);

/* ------------------------------------------------------------------------ */
/* (d) the compose folded into its adjacent products                         */
/* ------------------------------------------------------------------------ */

/* Bytes of workspace dora_compose_lora_fwd and dora_linear_fwd need (host
 * arithmetic; 0 for an invalid shape): s B split into two bf16 [out, r]
 * matrices.  dora_compose_lora_fwd_bf16 needs none. */
size_t dora_compose_fused_workspace(int64_t out, int64_t r);

/*
 * y = base + (g-1)*base + g*s*lora with lora = xa B^T computed in the same
 * kernel: the compose moved into the epilogue of the lora up-projection, so
 * lora never reaches memory (P1 ¶第二个创新是"融合Triton内核"技术 and
 * ¶从技术架构角度来看: the stable form, fp32 intermediates).  xa = x A^T is the
 * caller's down-projection.  s B is split into bf16 hi + lo (residual <= 2^-17
 * of s B), so each product is exact; fp32 accumulation on the tensor cores;
 * y is rounded once (nearest even) to bf16.
 *
 *   base  bf16 [T, out]   xa  bf16 [T, r]   y  bf16 [T, out]  (16-byte aligned)
 *   B     float32 [out, r] (4-byte aligned)   g  float32 [out] (16-byte aligned)
 *   workspace  >= dora_compose_fused_workspace(out, r) bytes, 256-byte aligned
 *   Sizes: T, out >= 0 (either 0 is a no-op), r >= 1; out % 8 == 0 and
 *   r % 8 == 0 (16-byte rows for the tensor-memory copies).
 * Two launches: the split of s B, then the fused kernel, as clusters of two
 * CTAs (one 256 x 256 tile of y per pair, tcgen05.mma.cta_group::2) where
 * the device can hold such clusters, else as single CTAs (128 x 256 tiles).
 * The fused kernel is a programmatic dependent launch on the split (its
 * set-up overlaps it); stream order is unchanged for the caller.
 * Results are bitwise reproducible for a given shape and device.
 */
dora_status dora_compose_lora_fwd(const void *base, const void *xa, const float *B,
                                  const float *g, float s,
                                  int64_t T, int64_t out, int64_t r, void *y,
                                  void *workspace, size_t workspace_bytes,
                                  dora_stream_t stream);

/*
 * The same lora up-projection form for a bf16 B (adapters kept in bf16):
 * y = base + (g-1)*base + g*(s*acc) with acc = xa B^T, B used as it is as the
 * tensor-core operand (every product exact in fp32, fp32 accumulation), s
 * applied to the accumulator in the epilogue, y rounded once to bf16
 * (P1 ¶第二个创新是"融合Triton内核"技术, the stable form).  One product instead
 * of the fp32-B form's two, and no split of B: one launch, no workspace.
 *
 *   base  bf16 [T, out]   xa  bf16 [T, r]   B  bf16 [out, r]   y  bf16 [T, out]
 *   g  float32 [out]; all five 16-byte aligned
 *   Sizes: T, out >= 0 (either 0 is a no-op), r >= 1; out % 8 == 0 and
 *   r % 8 == 0.
 * One launch (an ordinary one: it reads base from its first instruction), as
 * clusters of two CTAs where the device holds them, else single CTAs.
 * Results are bitwise reproducible for a given shape and device.
 */
dora_status dora_compose_lora_fwd_bf16(const void *base, const void *xa, const void *B,
                                       const float *g, float s,
                                       int64_t T, int64_t out, int64_t r, void *y,
                                       dora_stream_t stream);

/*
 * The whole layer output y = g*(x W0^T + s xa B^T) as ONE tensor-core GEMM
 * over K = in + r ([x | xa] times [W0 | s B]^T), with the compose in its
 * epilogue: neither base nor lora is formed.  x [T, in] and W0 [out, in] are
 * bf16 (16-byte aligned, in % 8 == 0); the rest as dora_compose_lora_fwd.
 * Since base + s lora stays in fp32 until the single rounding of y, this is the
 * page's stable evaluation with one rounding fewer.  Launches as
 * dora_compose_lora_fwd.
 */
dora_status dora_linear_fwd(const void *x, const void *W0, const void *xa, const float *B,
                            const float *g, float s,
                            int64_t T, int64_t in, int64_t out, int64_t r, void *y,
                            void *workspace, size_t workspace_bytes,
                            dora_stream_t stream);

/* ------------------------------------------------------------------------ */
/* diagnostics                                                               */
/* ------------------------------------------------------------------------ */

/*
 * Reads (synchronously: waits for the device) and clears the current device's
 * error word.  *code = 0 when no kernel gave up waiting; otherwise a nonzero
 * code naming the wait that timed out.  Returns DORA_ERR_DEVICE in that case.
 */
dora_status dora_device_error(int *code);

/* Number of kernels this process has launched through the library. */
uint64_t dora_kernel_launches(void);

/*
 * Testing hook for the failure path; no counterpart in the paper.  With on != 0
 * the tensor-core kernels of later dora_norm_factored, dora_norm_factored_bwd,
 * dora_compose_lora_fwd and dora_linear_fwd calls on the current device
 * withhold all their operand loads, so their bounded waits expire after
 * wait_limit_ns (0 = the default of 2 s): the kernels then record a code in the
 * device error word (see dora_device_error), free their tensor memory and
 * exit, leaving the context usable; their outputs are garbage.
 * on = 0 restores normal operation.  Synchronises the device.
 */
dora_status dora_test_stall_loads(int on, uint64_t wait_limit_ns);

/*
 * Testing hook; no counterpart in the paper.  With allow = 0, later
 * dora_compose_lora_fwd and dora_linear_fwd calls run their fused kernel as
 * single CTAs (128 x 256 tiles), as on a device that cannot hold clusters of
 * two; allow != 0 (the default) restores CTA pairs where the device has them.
 * Process-wide; never fails.
 */
dora_status dora_test_fused_pairs(int allow);

#ifdef __cplusplus
}
#endif

#endif /* DORA_H */
