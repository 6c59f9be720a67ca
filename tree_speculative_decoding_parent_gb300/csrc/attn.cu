// a4 tree-masked GQA attention: device-side split-KV scheduler, FP32 SIMT kernel,
// LSE combine, and the C-ABI entry point (bf16 goes to the tcgen05 kernel).
//
// Sources: "浙江大学、阿里巴巴联手破解AI推理瓶颈" §二 third gear (the flattened tree is verified
// in one parallel forward with tree position ids and an ancestor mask);
// "TreeGraft 精读：多起草器共嫁接一棵草稿树，让投机解码跨越快与好的单选题" §三 (tree-attention
// verification) and §七 (one target forward verifies the whole tree).
//
// Query rows of a segment (request b, KV head h) are ordered r = i*g + j for tree node i
// and query head h*g + j, so the g heads that share a KV head are adjacent. Key j of the
// segment is visible to node i when j < P (committed prefix) or when j = P + u and bit u
// of mask[b][i] is set (u an ancestor of i, or i itself).
#include <cuda_bf16.h>
#include <math.h>
#include <stdio.h>

#include <atomic>

#include "attn_common.cuh"
#include "attn_tc.cuh"
#include "gt_internal.cuh"
#include "launch.cuh"

namespace gt {

// ------------------------------------------------------------------------------------
// FP32 SIMT kernel (fp32 inputs; bf16 always runs on the tcgen05 kernel): CTA = (piece,
// group of 64 query rows); tiles of 64 keys in shared
// memory; S = Q K^T by 4x4 register blocks, masked online softmax (expf), O by 4x8 blocks.
// ------------------------------------------------------------------------------------
constexpr int SIMT_ROWS = 64, SIMT_KEYS = 64, SIMT_LD = 68, SIMT_SLD = 65;
constexpr size_t SIMT_SMEM =
    sizeof(float) * (2 * (size_t)ATTN_D * SIMT_LD + (size_t)SIMT_KEYS * ATTN_D +
                     (size_t)SIMT_ROWS * SIMT_SLD + 3 * SIMT_ROWS);


// Four consecutive fp32 elements (a 16-byte load; callers keep the element index a multiple
// of 4 and the base 16-byte aligned).
template <typename T> __device__ __forceinline__ float4 load4(const T *p);
template <> __device__ __forceinline__ float4 load4<float>(const float *p) {
  return *reinterpret_cast<const float4 *>(p);
}

template <typename T>
__global__ void __launch_bounds__(256)
attn_simt_kernel(const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V,
                 const uint64_t *__restrict__ mask, const int32_t *__restrict__ prefix_len,
                 const int32_t *__restrict__ n_nodes, int N, int Hq, int Hkv, int Lcap,
                 float scale, SchedArgs sa, AttnWs ws, int32_t *err) {
  pdl_enter();
  extern __shared__ float sm[];
  float *Qs = sm;                              // [d][SIMT_LD] (rows)
  float *Ks = Qs + ATTN_D * SIMT_LD;           // [d][SIMT_LD] (keys)
  float *Vs = Ks + ATTN_D * SIMT_LD;           // [keys][d]
  float *Ss = Vs + SIMT_KEYS * ATTN_D;         // [rows][SIMT_SLD]
  float *s_alpha = Ss + SIMT_ROWS * SIMT_SLD;  // [rows]
  float *s_m = s_alpha + SIMT_ROWS, *s_l = s_m + SIMT_ROWS;
  __shared__ uint64_t s_mask[SIMT_ROWS];

  const int p = blockIdx.x;
  int2 np;
  const int4 pc = schedule_piece(sa, p, ws, err, &np);
  if (pc.x < 0) return;
  const int seg = pc.x, b = seg / Hkv, h = seg - b * Hkv;
  const int g = Hq / Hkv;
  const int n = np.x, P = np.y, keys = P + n;  // from the schedule: no second load
  const int r0 = blockIdx.y * SIMT_ROWS;
  if (r0 >= g * n) return;
  const int tid = threadIdx.x;

  // Q rows (transposed into Qs), masks. Every load of a thread is issued before the first
  // store, so the tile costs one memory round trip, not one per element.
  constexpr int V4 = SIMT_ROWS * ATTN_D / 4 / 256;  // 4-element groups per thread (8)
  {
    float4 qv[V4];
#pragma unroll
    for (int k = 0; k < V4; ++k) {
      const int e4 = tid + k * 256, rl = e4 / (ATTN_D / 4), d4 = e4 - rl * (ATTN_D / 4);
      const int r = r0 + rl;
      qv[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < g * n) {
        const int i = r / g, hq = h * g + (r - i * g);
        qv[k] = load4<T>(Q + (((size_t)b * N + i) * Hq + hq) * ATTN_D + d4 * 4);
      }
    }
#pragma unroll
    for (int k = 0; k < V4; ++k) {
      const int e4 = tid + k * 256, rl = e4 / (ATTN_D / 4), d4 = e4 - rl * (ATTN_D / 4);
      Qs[(d4 * 4 + 0) * SIMT_LD + rl] = qv[k].x;
      Qs[(d4 * 4 + 1) * SIMT_LD + rl] = qv[k].y;
      Qs[(d4 * 4 + 2) * SIMT_LD + rl] = qv[k].z;
      Qs[(d4 * 4 + 3) * SIMT_LD + rl] = qv[k].w;
    }
  }
  if (tid < SIMT_ROWS) {
    const int r = r0 + tid;
    const uint64_t mrow = r < g * n ? mask[(size_t)b * N + r / g] : 0ull;
    s_mask[tid] = mrow;
    // checked builds: a tree row's mask holds the root and the node itself, no node past n
    GT_CHECKED(r >= g * n || (((mrow >> (r / g)) & 1ull) && (mrow & 1ull) &&
                              (n >= 64 || (mrow >> n) == 0ull)),
               err, GT_ERR_TREE);
  }

  const int ty = tid >> 4, tx = tid & 15;   // S / PV blocking
  const int srow = tid >> 2, spart = tid & 3;  // softmax: 4 threads per row
  float m_run = -INFINITY, l_run = 0.f;
  float acc[4][8];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[a][c] = 0.f;
  const size_t kv0 = ((size_t)b * Hkv + h) * Lcap;

  for (int tile = pc.y; tile < pc.z; ++tile) {
    const int kb = tile * SIMT_KEYS;
    __syncthreads();
    {
      constexpr int K4 = SIMT_KEYS * ATTN_D / 4 / 256;  // 4-element groups per thread (8)
      float4 kv[K4], vv[K4];
#pragma unroll
      for (int k = 0; k < K4; ++k) {
        const int e4 = tid + k * 256, c = e4 / (ATTN_D / 4), d4 = e4 - c * (ATTN_D / 4);
        const int j = kb + c;
        kv[k] = vv[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < keys) {
          kv[k] = load4<T>(K + (kv0 + j) * ATTN_D + d4 * 4);
          vv[k] = load4<T>(V + (kv0 + j) * ATTN_D + d4 * 4);
        }
      }
#pragma unroll
      for (int k = 0; k < K4; ++k) {
        const int e4 = tid + k * 256, c = e4 / (ATTN_D / 4), d4 = e4 - c * (ATTN_D / 4);
        Ks[(d4 * 4 + 0) * SIMT_LD + c] = kv[k].x;
        Ks[(d4 * 4 + 1) * SIMT_LD + c] = kv[k].y;
        Ks[(d4 * 4 + 2) * SIMT_LD + c] = kv[k].z;
        Ks[(d4 * 4 + 3) * SIMT_LD + c] = kv[k].w;
        *reinterpret_cast<float4 *>(Vs + c * ATTN_D + d4 * 4) = vv[k];
      }
    }
    __syncthreads();
    float s[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) s[a][c] = 0.f;
#pragma unroll 4
    for (int dd = 0; dd < ATTN_D; ++dd) {
      const float4 qv = *reinterpret_cast<const float4 *>(Qs + dd * SIMT_LD + ty * 4);
      const float4 kv = *reinterpret_cast<const float4 *>(Ks + dd * SIMT_LD + tx * 4);
      const float qa[4] = {qv.x, qv.y, qv.z, qv.w}, ka[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) s[a][c] = fmaf(qa[a], ka[c], s[a][c]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int rl = ty * 4 + a;
      const uint64_t mrow = s_mask[rl];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int j = kb + tx * 4 + c;
        bool vis = j < P;
        if (!vis && j < keys) vis = (mrow >> (j - P)) & 1ull;
        Ss[rl * SIMT_SLD + tx * 4 + c] = vis ? s[a][c] * scale : -INFINITY;
      }
    }
    __syncthreads();
    {  // online softmax of row srow over this tile
      float mx = -INFINITY;
      float* srow_p = Ss + srow * SIMT_SLD + spart * 16;
#pragma unroll
      for (int c = 0; c < 16; ++c) mx = fmaxf(mx, srow_p[c]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      const float alpha = (m_new == -INFINITY) ? 1.f : expf(m_run - m_new);
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float pv = (m_new == -INFINITY) ? 0.f : expf(srow_p[c] - m_new);
        srow_p[c] = pv;
        sum += pv;
      }
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      l_run = l_run * alpha + sum;
      m_run = m_new;
      if (spart == 0) s_alpha[srow] = alpha;
    }
    __syncthreads();
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float al = s_alpha[ty * 4 + a];
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[a][c] *= al;
    }
    for (int c = 0; c < SIMT_KEYS; ++c) {
      const float4 v0 = *reinterpret_cast<const float4 *>(Vs + c * ATTN_D + tx * 8);
      const float4 v1 = *reinterpret_cast<const float4 *>(Vs + c * ATTN_D + tx * 8 + 4);
      const float va[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const float pv = Ss[(ty * 4 + a) * SIMT_SLD + c];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[a][q] = fmaf(pv, va[q], acc[a][q]);
      }
    }
  }
  if (spart == 0) {
    s_m[srow] = m_run;
    s_l[srow] = l_run;
  }
  __syncthreads();
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int rl = ty * 4 + a, r = r0 + rl;
    if (r >= g * n) continue;
    const float l = s_l[rl];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float *dst = ws.opart + ((size_t)p * ws.rows_pad + r) * ATTN_D + tx * 8;
    *reinterpret_cast<float4 *>(dst) =
        make_float4(acc[a][0] * inv, acc[a][1] * inv, acc[a][2] * inv, acc[a][3] * inv);
    *reinterpret_cast<float4 *>(dst + 4) =
        make_float4(acc[a][4] * inv, acc[a][5] * inv, acc[a][6] * inv, acc[a][7] * inv);
    if (tx == 0) ws.lse[(size_t)p * ws.rows_pad + r] = l > 0.f ? s_m[rl] + logf(l) : -INFINITY;
  }
}

// ------------------------------------------------------------------------------------
// Combine: one warp per (b, i, query head); O = sum_p e^(lse_p - max) O_p / sum_p e^(...).
// ------------------------------------------------------------------------------------
template <typename T> __device__ __forceinline__ void store4(T *dst, float4 v);
template <> __device__ __forceinline__ void store4<float>(float *dst, float4 v) {
  *reinterpret_cast<float4 *>(dst) = v;
}
template <> __device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *dst, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), c = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t *>(&a);
  u.y = *reinterpret_cast<uint32_t *>(&c);
  *reinterpret_cast<uint2 *>(dst) = u;
}

// The merged output row w = (b, i, hq): the LSE-weighted sum of its segment's partial
// rows. Rows of nodes at or past n are zero. Returns false, having written nothing, when
// the flag *merge_flag (ws.hdr[1]; null: not read) says that no segment needs the combine.
template <typename T>
__device__ __forceinline__ bool combine_row(int w, int lane, const int32_t *__restrict__ n_nodes,
                                            int N, int Hq, int Hkv, const AttnWs &ws,
                                            T *__restrict__ O, bool direct_single,
                                            const int *merge_flag) {
  constexpr int PRE = 16;  // partials per lane loaded before any arithmetic
  const int hq = w % Hq, i = (w / Hq) % N, b = w / (Hq * N);
  const int g = Hq / Hkv, h = hq / g, r = i * g + (hq - h * g);
  T *dst = O + (size_t)w * ATTN_D + lane * 4;
  // the node count, the segment's pieces and (first row) the flag are independent loads:
  // the empty asm needs all three before the tests below, so they leave together instead
  // of the tests' branches holding the first two back
  const int n = n_nodes[b];
  int2 sg = ws.seg[b * Hkv + h];
  const int merge = merge_flag ? *merge_flag : 1;
  asm volatile("" ::"r"(n), "r"(sg.x), "r"(sg.y), "r"(merge));
  if (merge == 0) return false;
  if (direct_single && sg.y == 1) return true;  // written by the attention kernel
  if (i >= n) sg = make_int2(0, 0);  // rows past the tree are zero
  const size_t stride = (size_t)ws.rows_pad * ATTN_D;
  const float *src = ws.opart + ((size_t)sg.x * ws.rows_pad + r) * ATTN_D + lane * 4;
  // the first PRE partials and the log-sum-exps leave in one round trip
  float4 part[PRE];
#pragma unroll
  for (int j = 0; j < PRE; ++j)
    part[j] = j < sg.y ? *reinterpret_cast<const float4 *>(src + j * stride)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
  float mx = -INFINITY;
  for (int j = lane; j < sg.y; j += 32) mx = fmaxf(mx, ws.lse[(size_t)(sg.x + j) * ws.rows_pad + r]);
#pragma unroll
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (mx != -INFINITY) {
    float wsum = 0.f;
    for (int j0 = 0; j0 < sg.y; j0 += 32) {
      const int cnt = min(32, sg.y - j0);
      const float myw =
          lane < cnt ? expf(ws.lse[(size_t)(sg.x + j0 + lane) * ws.rows_pad + r] - mx) : 0.f;
      wsum += myw;
#pragma unroll 8
      for (int j = 0; j < cnt; ++j) {
        const float wt = __shfl_sync(0xffffffffu, myw, j);
        const int q = j0 + j;
        float4 v;
        if (q < PRE) {
#pragma unroll
          for (int u = 0; u < PRE; ++u)  // a register, not a local-memory index
            if (u == q) v = part[u];
        } else {
          v = *reinterpret_cast<const float4 *>(src + q * stride);
        }
        acc.x = fmaf(wt, v.x, acc.x);
        acc.y = fmaf(wt, v.y, acc.y);
        acc.z = fmaf(wt, v.z, acc.z);
        acc.w = fmaf(wt, v.w, acc.w);
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    const float inv = 1.f / wsum;
    acc = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
  store4<T>(dst, acc);
  return true;
}

// One warp per output row, grid-stride. direct_single: the attention kernel itself wrote
// the rows of segments that have exactly one piece (the tcgen05 kernel does), so those
// rows are skipped, and when no segment has another count (ws.hdr[1] == 0) the launch has
// nothing to do.
template <typename T>
__global__ void __launch_bounds__(256, 2)
attn_combine_kernel(const int32_t *__restrict__ n_nodes, int B, int N, int Hq, int Hkv,
                    AttnWs ws, T *__restrict__ O, int direct_single) {
  pdl_enter();
  const int rows = B * N * Hq, lane = threadIdx.x & 31;
  const int *flag = direct_single ? ws.hdr + 1 : nullptr;  // read with the first row only
  for (int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < rows;
       w += (gridDim.x * blockDim.x) >> 5) {
    if (!combine_row<T>(w, lane, n_nodes, N, Hq, Hkv, ws, O, direct_single != 0, flag)) return;
    flag = nullptr;
  }
}
static int device_sms() {
  static std::atomic<int> cache[64];  // per device; an SM count never changes
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 1024;  // conservative upper bound for the workspace size
  }
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0) {
    (void)cudaGetLastError();
    return 1024;
  }
  if (dev >= 0 && dev < 64) cache[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

// An array of `bytes` bytes at p must lie in device memory of device `dev` (a cudaMalloc-
// family allocation made there): the first and the last byte are looked up. The bf16
// kernel streams K and V through cluster-multicast TMA loads, which this library issues
// only over the memory of the GPU that runs the kernel, never over host, managed or peer
// memory; the same rule holds for every array of the call. Returns GT_ERR_ARG, with the
// detail for gt_last_error, otherwise.
static int check_own_device(const void *p, size_t bytes, int dev, const char *name) {
  const char *ends[2] = {static_cast<const char *>(p), static_cast<const char *>(p) + bytes - 1};
  for (const char *q : ends) {
    cudaPointerAttributes a{};
    const cudaError_t e = cudaPointerGetAttributes(&a, q);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      char msg[160];
      snprintf(msg, sizeof(msg), "gt_tree_attn: %s: cudaPointerGetAttributes: %s", name,
               cudaGetErrorString(e));
      note_message(msg);
      return GT_ERR_ARG;
    }
    if (a.type != cudaMemoryTypeDevice || a.device != dev) {
      char msg[160];
      snprintf(msg, sizeof(msg),
               "gt_tree_attn: %s is not device memory of the current device %d (memory type "
               "%d, device %d)",
               name, dev, (int)a.type, a.device);
      note_message(msg);
      return GT_ERR_ARG;
    }
  }
  return GT_OK;
}

static bool attn_args_ok(int B, int N, int Hq, int Hkv, int d, int Lcap) {
  return B >= 0 && N >= 1 && Hq >= 1 && Hkv >= 1 && d >= 1 && Lcap >= 1;
}
static bool attn_shape_ok(int N, int Hq, int Hkv, int d) {
  return d == ATTN_D && N <= ATTN_MAX_N && Hq % Hkv == 0 && (Hq / Hkv) * N <= 512;
}

}  // namespace gt

using namespace gt;

GT_API size_t gt_tree_attn_workspace(int B, int N, int Hq, int Hkv, int d, int Lcap) {
  if (!attn_args_ok(B, N, Hq, Hkv, d, Lcap) || !attn_shape_ok(N, Hq, Hkv, d)) return 0;
  const int S = B * Hkv;
  const int rows_pad = ceil_div((Hq / Hkv) * N, ATTN_ROWS_PAD) * ATTN_ROWS_PAD;
  return attn_ws_layout(nullptr, S, device_sms() + S, rows_pad, nullptr);
}

GT_API int gt_tree_attn(const void *Q, const void *K, const void *V, const uint64_t *mask,
                        const int32_t *prefix_len, const int32_t *n_nodes, int B, int N, int Hq,
                        int Hkv, int d, int Lcap, int dtype, float scale, void *O,
                        void *workspace, size_t ws_bytes, int32_t *err, gt_stream_t stream) {
  GT_TRACE("gt_tree_attn");
  if (!attn_args_ok(B, N, Hq, Hkv, d, Lcap)) return GT_ERR_ARG;
  if (dtype != GT_F32 && dtype != GT_BF16) return GT_ERR_ARG;
  if (!(scale > 0.f) || isinf(scale)) return GT_ERR_ARG;
  if (!attn_shape_ok(N, Hq, Hkv, d)) return GT_ERR_SHAPE;
  if (B == 0) return GT_OK;
  if (!Q || !K || !V || !mask || !prefix_len || !n_nodes || !O || !workspace) return GT_ERR_ARG;
  if (((uintptr_t)Q | (uintptr_t)K | (uintptr_t)V | (uintptr_t)O) & 15) return GT_ERR_ARG;
  if ((uintptr_t)workspace & 255) return GT_ERR_ARG;
  const int S = B * Hkv;
  if (S > 8192) return GT_ERR_SHAPE;
  {
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return launch_status(e, "cudaGetDevice");
    const size_t es = dtype == GT_BF16 ? 2 : 4;
    const size_t qo = (size_t)B * N * Hq * d * es, kv = (size_t)B * Hkv * Lcap * d * es;
    int rc = check_own_device(Q, qo, dev, "Q");
    if (rc == GT_OK) rc = check_own_device(K, kv, dev, "K");
    if (rc == GT_OK) rc = check_own_device(V, kv, dev, "V");
    if (rc == GT_OK) rc = check_own_device(O, qo, dev, "O");
    if (rc != GT_OK) return rc;
  }
  const int g = Hq / Hkv;
  const int rows_pad = ceil_div(g * N, ATTN_ROWS_PAD) * ATTN_ROWS_PAD;
  const int G = device_sms();
  AttnWs ws;
  const size_t need = attn_ws_layout(workspace, S, G + S, rows_pad, &ws);
  if (ws_bytes < need) return GT_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;

  // bf16 runs on the tcgen05 kernel for every supported shape, fp32 on the SIMT kernel
  const bool tc = dtype == GT_BF16;
  if (tc && !attn_tc_supported(g, N)) return GT_ERR_SHAPE;
  const int TK = tc ? ATTN_TC_KEYS : SIMT_KEYS;
  // the tcgen05 kernel runs one cluster per piece: aim for one wave of clusters
  const int Gs = tc ? attn_tc_pieces(g, N) : G;
  const SchedArgs sa{prefix_len, n_nodes, B, Hkv, N, Lcap, TK, Gs};
  // pieces the schedule can make: at most Gs while the segments are fewer than Gs (the
  // piece length is then searched so that they fit), else at most Gs + S. CTAs of pieces
  // past the schedule's count would only wait for an SM, find no work and exit.
  const int grid_pieces = S < Gs ? Gs : Gs + S;
  int rc;
  if (tc) {
    rc = attn_tc_launch(Q, K, V, mask, sa, B, N, Hq, Hkv, Lcap, scale, ws, grid_pieces, O, err,
                        s);
  } else {
    static SmemAttr attr_f32;
    rc = ensure_smem(attn_simt_kernel<float>, (int)SIMT_SMEM, attr_f32,
                     "cudaFuncSetAttribute(attn_simt_kernel)");
    if (rc != GT_OK) return rc;
    rc = launch(attn_simt_kernel<float>, dim3(grid_pieces, ceil_div(g * N, SIMT_ROWS)), dim3(256),
                SIMT_SMEM, s, (const float *)Q, (const float *)K, (const float *)V, mask,
                prefix_len, n_nodes, N, Hq, Hkv, Lcap, scale, sa, ws, err);
  }
  if (rc != GT_OK) return rc;
  // a warp per output row, at most two CTAs of 8 warps per SM (one resident wave)
  const int warps = B * N * Hq;
  const dim3 cgrid(max(1, min(ceil_div(warps, 8), 2 * G)));
  if (dtype == GT_F32)
    return launch(attn_combine_kernel<float>, cgrid, dim3(256), 0, s, n_nodes, B, N, Hq, Hkv, ws,
                  (float *)O, 0);
  return launch(attn_combine_kernel<__nv_bfloat16>, cgrid, dim3(256), 0, s, n_nodes, B, N, Hq,
                Hkv, ws, (__nv_bfloat16 *)O, tc ? 1 : 0);
}
