// Fused DoRA compose, forward and backward, for GB300 (sm_103a).
//
// Method source: web page "人工智能训练新突破：Anthropic团队破解大模型微调内存瓶颈难题"
// (techwalker.com), paragraphs on the fused kernel (four elementwise passes
// fused into one), on numerical stability near g = 1 (the form
// (g-1)*base + g*s*lora with fp32 intermediates) and on the fused backward
// and its d_mag reduction order.
//
// Both directions are one streaming pass over [T, out] and are bound by HBM
// bandwidth.  Thread layout: a 256-thread block is 32 column groups x 8 token
// lanes.  A column group is VEC consecutive columns read with one 128-bit
// access (VEC = 8 for bf16, 4 for fp32; VEC = 1 on the scalar path for ragged
// or unaligned rows).  A warp is one token row of 32 groups, i.e. 512
// contiguous bytes for bf16.  Per-column constants (g-1, g*s) stay in
// registers; each thread walks tokens t = t0, t0 + lanes, ... where lanes =
// 8 * gridDim.y, so the grid is sized to the device (SM count x resident
// blocks) and not to T.
//
// d_mag is reduced without atomics in a fixed order: each thread sums its
// own tokens in increasing t, the 8 lanes of a block are summed in lane order
// through shared memory into one partial row per blockIdx.y, and a second
// kernel sums those rows in increasing blockIdx.y and divides by the norm.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"

namespace {

constexpr int kBX = 32;     // column groups per block
constexpr int kBY = 8;      // token lanes per block
constexpr int kThreads = kBX * kBY;
constexpr int kMaxSMs = 256;             // workspace bound: any device up to this size
constexpr int kMaxBlocksPerSM = 2048 / kThreads;

// ---------------------------------------------------------------------------
// Vector I/O: Raw is what one access moves; unpack/pack convert to fp32.
// ---------------------------------------------------------------------------
template <typename Act, int VEC> struct Io;

template <> struct Io<__nv_bfloat16, 8> {
  using Raw = uint4;
  static __device__ __forceinline__ Raw load(const __nv_bfloat16 *p, int64_t e) {
    return __ldcs(reinterpret_cast<const uint4 *>(p + e));
  }
  static __device__ __forceinline__ void store(__nv_bfloat16 *p, int64_t e, Raw r) {
    __stcs(reinterpret_cast<uint4 *>(p + e), r);
  }
  static __device__ __forceinline__ void unpack(Raw r, float (&v)[8]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = __uint_as_float(w[k] << 16);
      v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ Raw pack(const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
      w[k] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <> struct Io<float, 4> {
  using Raw = float4;
  static __device__ __forceinline__ Raw load(const float *p, int64_t e) {
    return __ldcs(reinterpret_cast<const float4 *>(p + e));
  }
  static __device__ __forceinline__ void store(float *p, int64_t e, Raw r) {
    __stcs(reinterpret_cast<float4 *>(p + e), r);
  }
  static __device__ __forceinline__ void unpack(Raw r, float (&v)[4]) {
    v[0] = r.x; v[1] = r.y; v[2] = r.z; v[3] = r.w;
  }
  static __device__ __forceinline__ Raw pack(const float (&v)[4]) { return make_float4(v[0], v[1], v[2], v[3]); }
};

template <> struct Io<__nv_bfloat16, 1> {
  using Raw = unsigned short;
  static __device__ __forceinline__ Raw load(const __nv_bfloat16 *p, int64_t e) {
    return __ldcs(reinterpret_cast<const unsigned short *>(p + e));
  }
  static __device__ __forceinline__ void store(__nv_bfloat16 *p, int64_t e, Raw r) {
    __stcs(reinterpret_cast<unsigned short *>(p + e), r);
  }
  static __device__ __forceinline__ void unpack(Raw r, float (&v)[1]) { v[0] = __uint_as_float(uint32_t(r) << 16); }
  static __device__ __forceinline__ Raw pack(const float (&v)[1]) {
    __nv_bfloat16 h = __float2bfloat16_rn(v[0]);
    return *reinterpret_cast<unsigned short *>(&h);
  }
};

template <> struct Io<float, 1> {
  using Raw = float;
  static __device__ __forceinline__ Raw load(const float *p, int64_t e) { return __ldcs(p + e); }
  static __device__ __forceinline__ void store(float *p, int64_t e, Raw r) { __stcs(p + e, r); }
  static __device__ __forceinline__ void unpack(Raw r, float (&v)[1]) { v[0] = r; }
  static __device__ __forceinline__ Raw pack(const float (&v)[1]) { return v[0]; }
};

// ---------------------------------------------------------------------------
// forward: y = base + ((g-1)*base + (g*s)*lora), fp32, one rounding at the store
// ---------------------------------------------------------------------------
template <typename Act, int VEC>
__global__ void __launch_bounds__(kThreads)
compose_fwd_kernel(const Act *__restrict__ base, const Act *__restrict__ lora,
                   const float *__restrict__ g, float s, int64_t T, int64_t out,
                   Act *__restrict__ y) {
  using IO = Io<Act, VEC>;
  using Raw = typename IO::Raw;
  constexpr int U = 4;  // token rows in flight per thread
  const int64_t ncg = out / VEC;
  const int64_t cg = (int64_t)blockIdx.x * kBX + threadIdx.x;
  if (cg >= ncg) return;
  const int64_t lanes = (int64_t)gridDim.y * kBY;
  const int64_t c0 = cg * VEC;

  float gm1[VEC], gs[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) {
    const float gv = __ldg(g + c0 + v);
    gm1[v] = gv - 1.0f;
    gs[v] = gv * s;
  }

  int64_t t = (int64_t)blockIdx.y * kBY + threadIdx.y;
  for (; t + (U - 1) * lanes < T; t += U * lanes) {
    Raw rb[U], rl[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t e = (t + u * lanes) * out + c0;
      rb[u] = IO::load(base, e);
      rl[u] = IO::load(lora, e);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float b[VEC], l[VEC];
      IO::unpack(rb[u], b);
      IO::unpack(rl[u], l);
#pragma unroll
      for (int v = 0; v < VEC; ++v) b[v] = b[v] + fmaf(gm1[v], b[v], gs[v] * l[v]);
      IO::store(y, (t + u * lanes) * out + c0, IO::pack(b));
    }
  }
  for (; t < T; t += lanes) {
    const int64_t e = t * out + c0;
    float b[VEC], l[VEC];
    IO::unpack(IO::load(base, e), b);
    IO::unpack(IO::load(lora, e), l);
#pragma unroll
    for (int v = 0; v < VEC; ++v) b[v] = b[v] + fmaf(gm1[v], b[v], gs[v] * l[v]);
    IO::store(y, e, IO::pack(b));
  }
}

// ---------------------------------------------------------------------------
// backward: d_base = g*dy, d_lora = (g*s)*dy, partial d_mag sums
// ---------------------------------------------------------------------------
template <typename Act, int VEC>
__global__ void __launch_bounds__(kThreads)
compose_bwd_kernel(const Act *__restrict__ dy, const Act *__restrict__ base,
                   const Act *__restrict__ lora, const float *__restrict__ g, float s,
                   int64_t T, int64_t out, Act *__restrict__ d_base,
                   Act *__restrict__ d_lora, float *__restrict__ part) {
  using IO = Io<Act, VEC>;
  using Raw = typename IO::Raw;
  constexpr int U = 2;
  __shared__ float red[kBY][kBX * VEC];

  const int64_t ncg = out / VEC;
  const int64_t cg = (int64_t)blockIdx.x * kBX + threadIdx.x;
  const bool active = cg < ncg;
  const int64_t lanes = (int64_t)gridDim.y * kBY;
  const int64_t c0 = cg * VEC;

  float acc[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) acc[v] = 0.0f;

  if (active) {
    float gg[VEC], gs[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      gg[v] = __ldg(g + c0 + v);
      gs[v] = gg[v] * s;
    }
    int64_t t = (int64_t)blockIdx.y * kBY + threadIdx.y;
    for (; t + (U - 1) * lanes < T; t += U * lanes) {
      Raw rd[U], rb[U], rl[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t e = (t + u * lanes) * out + c0;
        rd[u] = IO::load(dy, e);
        rb[u] = IO::load(base, e);
        rl[u] = IO::load(lora, e);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float d[VEC], b[VEC], l[VEC], ob[VEC], ol[VEC];
        IO::unpack(rd[u], d);
        IO::unpack(rb[u], b);
        IO::unpack(rl[u], l);
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
          ob[v] = gg[v] * d[v];
          ol[v] = gs[v] * d[v];
          acc[v] = fmaf(d[v], fmaf(s, l[v], b[v]), acc[v]);
        }
        const int64_t e = (t + u * lanes) * out + c0;
        IO::store(d_base, e, IO::pack(ob));
        IO::store(d_lora, e, IO::pack(ol));
      }
    }
    for (; t < T; t += lanes) {
      const int64_t e = t * out + c0;
      float d[VEC], b[VEC], l[VEC], ob[VEC], ol[VEC];
      IO::unpack(IO::load(dy, e), d);
      IO::unpack(IO::load(base, e), b);
      IO::unpack(IO::load(lora, e), l);
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        ob[v] = gg[v] * d[v];
        ol[v] = gs[v] * d[v];
        acc[v] = fmaf(d[v], fmaf(s, l[v], b[v]), acc[v]);
      }
      IO::store(d_base, e, IO::pack(ob));
      IO::store(d_lora, e, IO::pack(ol));
    }
  }

  // fixed-order sum of the 8 token lanes of this block
#pragma unroll
  for (int v = 0; v < VEC; ++v) red[threadIdx.y][threadIdx.x * VEC + v] = acc[v];
  __syncthreads();
  if (threadIdx.y == 0 && active) {
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      float sum = red[0][threadIdx.x * VEC + v];
#pragma unroll
      for (int k = 1; k < kBY; ++k) sum += red[k][threadIdx.x * VEC + v];
      part[(int64_t)blockIdx.y * out + c0 + v] = sum;
    }
  }
}

// d_mag[j] = (sum over partial rows in increasing order) / norm[j]
__global__ void __launch_bounds__(256)
dmag_reduce_kernel(const float *__restrict__ part, int64_t rows, int64_t out,
                   const float *__restrict__ norm, float *__restrict__ d_mag) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= out) return;
  float sum = 0.0f;
  int64_t k = 0;
  for (; k + 4 <= rows; k += 4) {
    const float a0 = part[(k + 0) * out + j], a1 = part[(k + 1) * out + j];
    const float a2 = part[(k + 2) * out + j], a3 = part[(k + 3) * out + j];
    sum += a0;
    sum += a1;
    sum += a2;
    sum += a3;
  }
  for (; k < rows; ++k) sum += part[k * out + j];
  d_mag[j] = sum / norm[j];
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
struct Occ {
  int blocks_per_sm = 0;
};

template <typename K>
int blocks_per_sm(K kernel, int device) {
  static std::mutex mu;
  static int cache[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return 1;
  if (cache[device] == 0) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kThreads, 0) != cudaSuccess || b <= 0) b = 1;
    cache[device] = b;
  }
  return cache[device];
}

struct Grid {
  int64_t gx, gy;
};

Grid plan_grid(int64_t T, int64_t ncg, int64_t target_blocks) {
  Grid gr;
  gr.gx = dora::ceil_div(ncg, kBX);
  // as many grid rows as the resident blocks fill, rounded DOWN: every block
  // has the same work, so a block beyond the resident ones would run alone
  // in a second wave (bf16, out = 14336 on 152 SMs x 4 blocks: 56 x 11 = 616
  // blocks took 269 us for the forward at T = 16384, 56 x 10 take 215 us)
  int64_t gy = target_blocks / gr.gx;
  const int64_t gy_max = dora::ceil_div(T, kBY);
  if (gy > gy_max) gy = gy_max;
  if (gy < 1) gy = 1;
  if (gy > 65535) gy = 65535;
  gr.gy = gy;
  return gr;
}

int64_t bwd_rows_bound(int64_t T, int64_t out) {
  // the widest vector (8 bf16) gives the fewest column groups and so the
  // most grid rows; any narrower path launches no more rows than this
  const int64_t gx_min = dora::ceil_div(dora::ceil_div(out, 8), kBX);
  Grid gr = plan_grid(T, gx_min * kBX, (int64_t)kMaxSMs * kMaxBlocksPerSM);
  return gr.gy;
}

bool valid_dtype(dora_dtype act) { return act == DORA_F32 || act == DORA_BF16; }

template <typename Act>
bool vector_ok(int64_t out, std::initializer_list<const void *> ptrs) {
  constexpr int vec = 16 / sizeof(Act);
  if (out % vec != 0) return false;
  for (const void *p : ptrs)
    if (!dora::aligned(p, 16)) return false;
  return true;
}

template <typename Act, int VEC>
dora_status launch_fwd(const void *base, const void *lora, const float *g, float s, int64_t T,
                       int64_t out, void *y, cudaStream_t stream, int device, int sms) {
  auto kern = compose_fwd_kernel<Act, VEC>;
  const int bps = blocks_per_sm(kern, device);
  Grid gr = plan_grid(T, out / VEC, (int64_t)sms * bps);
  kern<<<dim3((unsigned)gr.gx, (unsigned)gr.gy), dim3(kBX, kBY), 0, stream>>>(
      static_cast<const Act *>(base), static_cast<const Act *>(lora), g, s, T, out, static_cast<Act *>(y));
  dora::count_launches(1);
  return dora::launch_status();
}

template <typename Act, int VEC>
dora_status launch_bwd(const void *dy, const void *base, const void *lora, const float *g,
                       const float *norm, float s, int64_t T, int64_t out, void *d_base, void *d_lora,
                       float *d_mag, float *part, size_t part_bytes, cudaStream_t stream, int device,
                       int sms) {
  auto kern = compose_bwd_kernel<Act, VEC>;
  const int bps = blocks_per_sm(kern, device);
  int64_t rows = 0;
  if (T > 0) {
    Grid gr = plan_grid(T, out / VEC, (int64_t)sms * bps);
    rows = gr.gy;
    if ((size_t)rows * (size_t)out * sizeof(float) > part_bytes) return DORA_ERR_WORKSPACE;
    kern<<<dim3((unsigned)gr.gx, (unsigned)gr.gy), dim3(kBX, kBY), 0, stream>>>(
        static_cast<const Act *>(dy), static_cast<const Act *>(base), static_cast<const Act *>(lora), g, s, T,
        out, static_cast<Act *>(d_base), static_cast<Act *>(d_lora), part);
    dora::count_launches(1);
    if (cudaGetLastError() != cudaSuccess) return DORA_ERR_CUDA;
  }
  dmag_reduce_kernel<<<(unsigned)dora::ceil_div(out, 256), 256, 0, stream>>>(part, rows, out, norm, d_mag);
  dora::count_launches(1);
  return dora::launch_status();
}

}  // namespace

extern "C" dora_status dora_compose_fwd(dora_dtype act, const void *base, const void *lora,
                                        const float *g, float s, int64_t T, int64_t out, void *y,
                                        dora_stream_t stream) {
  if (!valid_dtype(act)) return DORA_ERR_DTYPE;
  if (T < 0 || out < 0) return DORA_ERR_SHAPE;
  if (T == 0 || out == 0) return DORA_OK;
  if (!base || !lora || !g || !y) return DORA_ERR_NULL;
  const size_t esz = act == DORA_F32 ? 4 : 2;
  if (!dora::aligned(base, esz) || !dora::aligned(lora, esz) || !dora::aligned(y, esz) || !dora::aligned(g, 4))
    return DORA_ERR_ALIGN;
  dora::DeviceInfo info;
  int device = 0;
  dora_status st = dora::current_device(&info, &device);
  if (st != DORA_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (act == DORA_BF16) {
    if (vector_ok<__nv_bfloat16>(out, {base, lora, y}))
      return launch_fwd<__nv_bfloat16, 8>(base, lora, g, s, T, out, y, cs, device, info.sms);
    return launch_fwd<__nv_bfloat16, 1>(base, lora, g, s, T, out, y, cs, device, info.sms);
  }
  if (vector_ok<float>(out, {base, lora, y}))
    return launch_fwd<float, 4>(base, lora, g, s, T, out, y, cs, device, info.sms);
  return launch_fwd<float, 1>(base, lora, g, s, T, out, y, cs, device, info.sms);
}

extern "C" size_t dora_compose_bwd_workspace(int64_t T, int64_t out) {
  if (T < 0 || out < 0) return 0;
  if (out == 0) return 0;
  if (T == 0) return 256;
  return (size_t)bwd_rows_bound(T, out) * (size_t)out * sizeof(float);
}

extern "C" dora_status dora_compose_bwd(dora_dtype act, const void *grad_out, const void *base,
                                        const void *lora, const float *g, const float *norm, float s,
                                        int64_t T, int64_t out, void *d_base, void *d_lora, float *d_mag,
                                        void *workspace, size_t workspace_bytes, dora_stream_t stream) {
  if (!valid_dtype(act)) return DORA_ERR_DTYPE;
  if (T < 0 || out < 0) return DORA_ERR_SHAPE;
  if (out == 0) return DORA_OK;
  if (!g || !norm || !d_mag) return DORA_ERR_NULL;
  if (T > 0 && (!grad_out || !base || !lora || !d_base || !d_lora)) return DORA_ERR_NULL;
  if (!workspace) return DORA_ERR_WORKSPACE;
  if (!dora::aligned(workspace, 256) || workspace_bytes < dora_compose_bwd_workspace(T, out))
    return DORA_ERR_WORKSPACE;
  const size_t esz = act == DORA_F32 ? 4 : 2;
  if (T > 0 && (!dora::aligned(grad_out, esz) || !dora::aligned(base, esz) || !dora::aligned(lora, esz) ||
                !dora::aligned(d_base, esz) || !dora::aligned(d_lora, esz)))
    return DORA_ERR_ALIGN;
  if (!dora::aligned(g, 4) || !dora::aligned(norm, 4) || !dora::aligned(d_mag, 4)) return DORA_ERR_ALIGN;
  dora::DeviceInfo info;
  int device = 0;
  dora_status st = dora::current_device(&info, &device);
  if (st != DORA_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  float *part = static_cast<float *>(workspace);
  if (act == DORA_BF16) {
    if (vector_ok<__nv_bfloat16>(out, {grad_out, base, lora, d_base, d_lora}))
      return launch_bwd<__nv_bfloat16, 8>(grad_out, base, lora, g, norm, s, T, out, d_base, d_lora, d_mag, part,
                                          workspace_bytes, cs, device, info.sms);
    return launch_bwd<__nv_bfloat16, 1>(grad_out, base, lora, g, norm, s, T, out, d_base, d_lora, d_mag, part,
                                        workspace_bytes, cs, device, info.sms);
  }
  if (vector_ok<float>(out, {grad_out, base, lora, d_base, d_lora}))
    return launch_bwd<float, 4>(grad_out, base, lora, g, norm, s, T, out, d_base, d_lora, d_mag, part,
                                workspace_bytes, cs, device, info.sms);
  return launch_bwd<float, 1>(grad_out, base, lora, g, norm, s, T, out, d_base, d_lora, d_mag, part,
                              workspace_bytes, cs, device, info.sms);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of the backward.
//
// Some callers cannot allocate device memory at the point where they run the
// backward: code embedded in a host application that owns a fixed device
// memory pool and hands out no allocator, or services that forbid cudaMalloc
// after start-up because it synchronises the device and fragments memory that
// is shared with other work.  For them the d_mag partial sums live in one
// file-scope device array of fixed size instead of a caller workspace.  Every
// GPU that loads the library holds this array until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr int64_t kNoAllocScratchFloats = DORA_NOALLOC_SCRATCH_FLOATS;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

// Device address of g_noalloc_scratch, looked up once per device (and again
// after a device reset, which gives the device a new context and reloads the
// module) with that device current.  In host code the symbol name is only a
// host-side stand-in, never a device address.
float *noalloc_scratch_address(int device) {
  static std::mutex mu;
  static float *addr[64] = {};
  static uint64_t ctx_of[64] = {};
  if (device < 0 || device >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  const uint64_t ctx = dora::context_id();
  if (!addr[device] || ctx == 0 || ctx != ctx_of[device]) {
    addr[device] = nullptr;
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[device] = static_cast<float *>(ptr);
    ctx_of[device] = dora::context_id();
  }
  return addr[device];
}

template <typename Act, int VEC>
dora_status launch_bwd_noalloc(const void *dy, const void *base, const void *lora, const float *g,
                               const float *norm, float s, int64_t T, int64_t out, void *d_base, void *d_lora,
                               float *d_mag, float *part, cudaStream_t stream, int device, int sms) {
  auto kern = compose_bwd_kernel<Act, VEC>;
  const int bps = blocks_per_sm(kern, device);
  int64_t rows = 0;
  if (T > 0) {
    const Grid gr = plan_grid(T, out / VEC, (int64_t)sms * bps);
    // The grid plan keeps rows * out below 2 x (SMs x resident blocks) x 32 x
    // VEC <= SMs x 4096 floats (at most 8 resident blocks of 256 threads,
    // VEC <= 8): under 2^20 on any device with up to 256 SMs (GB300 has 152),
    // so the partial rows always fit the scratch.  Checked anyway, and refused
    // rather than launched with a different summation order.
    if (gr.gy * out > kNoAllocScratchFloats) return DORA_ERR_SHAPE;
    rows = gr.gy;
    kern<<<dim3((unsigned)gr.gx, (unsigned)gr.gy), dim3(kBX, kBY), 0, stream>>>(
        static_cast<const Act *>(dy), static_cast<const Act *>(base), static_cast<const Act *>(lora), g, s, T,
        out, static_cast<Act *>(d_base), static_cast<Act *>(d_lora), part);
    dora::count_launches(1);
    if (cudaGetLastError() != cudaSuccess) return DORA_ERR_CUDA;
  }
  dmag_reduce_kernel<<<(unsigned)dora::ceil_div(out, 256), 256, 0, stream>>>(part, rows, out, norm, d_mag);
  dora::count_launches(1);
  return dora::launch_status();
}

}  // namespace

extern "C" dora_status dora_compose_bwd_noalloc(dora_dtype act, const void *grad_out, const void *base,
                                                const void *lora, const float *g, const float *norm, float s,
                                                int64_t T, int64_t out, void *d_base, void *d_lora, float *d_mag,
                                                dora_stream_t stream) {
  if (!valid_dtype(act)) return DORA_ERR_DTYPE;
  if (T < 0 || out < 0) return DORA_ERR_SHAPE;
  if (out > kNoAllocScratchFloats) return DORA_ERR_SHAPE;   // one partial row must fit the scratch
  if (out == 0) return DORA_OK;
  if (!g || !norm || !d_mag) return DORA_ERR_NULL;
  if (T > 0 && (!grad_out || !base || !lora || !d_base || !d_lora)) return DORA_ERR_NULL;
  const size_t esz = act == DORA_F32 ? 4 : 2;
  if (T > 0 && (!dora::aligned(grad_out, esz) || !dora::aligned(base, esz) || !dora::aligned(lora, esz) ||
                !dora::aligned(d_base, esz) || !dora::aligned(d_lora, esz)))
    return DORA_ERR_ALIGN;
  if (!dora::aligned(g, 4) || !dora::aligned(norm, 4) || !dora::aligned(d_mag, 4)) return DORA_ERR_ALIGN;
  dora::DeviceInfo info;
  int device = 0;
  dora_status st = dora::current_device(&info, &device);
  if (st != DORA_OK) return st;
  float *part = noalloc_scratch_address(device);
  if (!part) return DORA_ERR_CUDA;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (act == DORA_BF16) {
    if (vector_ok<__nv_bfloat16>(out, {grad_out, base, lora, d_base, d_lora}))
      return launch_bwd_noalloc<__nv_bfloat16, 8>(grad_out, base, lora, g, norm, s, T, out, d_base, d_lora, d_mag,
                                                  part, cs, device, info.sms);
    return launch_bwd_noalloc<__nv_bfloat16, 1>(grad_out, base, lora, g, norm, s, T, out, d_base, d_lora, d_mag,
                                                part, cs, device, info.sms);
  }
  if (vector_ok<float>(out, {grad_out, base, lora, d_base, d_lora}))
    return launch_bwd_noalloc<float, 4>(grad_out, base, lora, g, norm, s, T, out, d_base, d_lora, d_mag, part, cs,
                                        device, info.sms);
  return launch_bwd_noalloc<float, 1>(grad_out, base, lora, g, norm, s, T, out, d_base, d_lora, d_mag, part, cs,
                                      device, info.sms);
}
