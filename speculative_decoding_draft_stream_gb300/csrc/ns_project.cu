// Dense head on a row range of W_head: logits[r, j] = sum_h hidden[r, h] *
// W_head[j, h] for j < rows (MicroSpec §3.1 Eq. 1 over the whole vocabulary,
// or over a static first-rows sub-head) and the per-row top-k with ids = row
// numbers.  These are the comparators of the dynamic sub-head, whose own
// projection runs in the fused tcgen05 kernel.
//
// Projection kernel.  A tile is 64 W_head rows x 64 hidden rows; the K loop
// streams 64-wide k slices of both operands through a 4-stage cp.async
// pipeline into 128-byte-swizzled shared memory, and four warps each
// multiply 16 rows against all 64 hidden rows with bf16 tensor-core MMAs
// (mma.sync, fp32 accumulate).  The grid is fixed (two CTAs per SM); when
// there are fewer tiles than CTAs, K is split S ways, partial tiles go to
// scratch, and the last CTA of a tile to arrive adds them in split order
// (deterministic).
#include "ns_internal.cuh"

namespace ns {
namespace {

constexpr int kStageBytesA = kProjBM * kProjBK * 2;  // 8 KB
constexpr int kStageBytesB = kProjBN * kProjBK * 2;  // 8 KB
constexpr int kStageBytes = kStageBytesA + kStageBytesB;
constexpr int kTilePitch = kProjBM + 4;  // floats per hidden row of the staged output tile
constexpr int kTileFloats = kProjBN * kProjBM;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk c of row r in a [rows x 128 B] swizzled stage.
__device__ __forceinline__ int swz(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

__global__ void __launch_bounds__(kProjThreads) project_kernel(ProjArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m = a.rows_host;
  const int T = (m + kProjBM - 1) / kProjBM;
  if (T == 0) return;
  const int KC = a.H / kProjBK;
  int S = 1;
  if (T < (int)gridDim.x) {
    S = (int)gridDim.x / T;
    S = S < kProjMaxSplit ? S : kProjMaxSplit;
    S = S < KC ? S : KC;
  }
  const int total = T * S;
  const int c = tid & 7;  // 16-byte chunk column this thread loads
  const int g = lane >> 2, tq = lane & 3;

  for (int w = blockIdx.x; w < total; w += gridDim.x) {
    const int t = w / S, sp = w - t * S;
    const int kc0 = sp * KC / S, kc1 = (sp + 1) * KC / S, nk = kc1 - kc0;
    const int row0 = t * kProjBM;

    const uint16_t *asrc[4];
    const uint16_t *bsrc[4];
    uint32_t abytes[4], bbytes[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = (tid >> 3) + 16 * q;
      const int j = row0 + r;
      const bool av = j < m;
      asrc[q] = a.rows + (size_t)(av ? j : 0) * a.H + c * 8;
      abytes[q] = av ? 16u : 0u;
      const bool bv = r < a.n;
      bsrc[q] = a.hid + (size_t)(bv ? r : 0) * a.H + c * 8;
      bbytes[q] = bv ? 16u : 0u;
    }
    auto load_stage = [&](int kt, int slot) {
      const int koff = (kc0 + kt) * kProjBK;
      uint8_t *As = smem + slot * kStageBytes;
      uint8_t *Bs = As + kStageBytesA;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = (tid >> 3) + 16 * q;
        cp_async16(smem_addr(As + swz(r, c)), asrc[q] + koff, abytes[q]);
        cp_async16(smem_addr(Bs + swz(r, c)), bsrc[q] + koff, bbytes[q]);
      }
    };

    float acc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;

#pragma unroll
    for (int st = 0; st < kProjStages - 1; ++st) {
      if (st < nk) load_stage(st, st);
      cp_async_commit();
    }
    for (int kt = 0; kt < nk; ++kt) {
      cp_async_wait<kProjStages - 2>();
      __syncthreads();
      const int slot = kt % kProjStages;
      const uint8_t *As = smem + slot * kStageBytes;
      const uint8_t *Bs = As + kStageBytesA;
#pragma unroll
      for (int kk = 0; kk < kProjBK / 16; ++kk) {
        uint32_t af[4];
        {
          const int mi = lane >> 3;
          const int r = warp * 16 + (mi & 1) * 8 + (lane & 7);
          ldsm_x4(smem_addr(As + swz(r, kk * 2 + (mi >> 1))), af[0], af[1], af[2], af[3]);
        }
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int mi = lane >> 3;
          const int r = 16 * p + (mi >> 1) * 8 + (lane & 7);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_addr(Bs + swz(r, kk * 2 + (mi & 1))), b0, b1, b2, b3);
          mma_16816(acc[2 * p], af, b0, b1);
          mma_16816(acc[2 * p + 1], af, b2, b3);
        }
      }
      const int nxt = kt + kProjStages - 1;
      if (nxt < nk) load_stage(nxt, nxt % kProjStages);
      cp_async_commit();
    }
    cp_async_wait<0>();
    __syncthreads();

    // Stage the tile as tile[r][j] (r = hidden row, j = W row within the tile).
    float *tile = reinterpret_cast<float *>(smem);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int jl = warp * 16 + g + (e >= 2 ? 8 : 0);
        const int r = 8 * nt + 2 * tq + (e & 1);
        tile[r * kTilePitch + jl] = acc[nt][e];
      }
    __syncthreads();

    if (S == 1) {
      for (int i = tid; i < a.n * kProjBM; i += kProjThreads) {
        const int r = i / kProjBM, jl = i - r * kProjBM;
        const int j = row0 + jl;
        if (j < m) a.logits[(size_t)r * a.ld + j] = tile[r * kTilePitch + jl];
      }
    } else {
      float *part = a.part + (size_t)w * kTileFloats;
      for (int i = tid; i < kProjBN * (kProjBM / 4); i += kProjThreads) {
        const int r = i >> 4, j4 = i & 15;
        const float4 v = *reinterpret_cast<const float4 *>(tile + r * kTilePitch + 4 * j4);
        __stcg(reinterpret_cast<float4 *>(part + r * kProjBM + 4 * j4), v);
      }
      __threadfence();
      __syncthreads();
      if (tid == 0) s_last = (atomicAdd(a.tickets + t, 1) == S - 1);
      __syncthreads();
      if (s_last) {
        __threadfence();
        if (tid == 0) a.tickets[t] = 0;
        const float *base = a.part + (size_t)t * S * kTileFloats;
        for (int i = tid; i < a.n * (kProjBM / 4); i += kProjThreads) {
          const int r = i >> 4, j4 = i & 15;
          const int o = r * kProjBM + 4 * j4;
          float4 s4 = __ldcg(reinterpret_cast<const float4 *>(base + o));
          for (int s2 = 1; s2 < S; ++s2) {
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(base + (size_t)s2 * kTileFloats + o));
            s4.x += v.x;
            s4.y += v.y;
            s4.z += v.z;
            s4.w += v.w;
          }
          const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = row0 + 4 * j4 + e;
            if (j < m) a.logits[(size_t)r * a.ld + j] = sv[e];
          }
        }
      }
    }
    __syncthreads();
  }
}

// Per-row top-k over logits[r, 0:m): one CTA per hidden row.  Column j stands
// for global id idmap[j] when idmap is given, else for j itself.
template <int KMAX>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float *logits, int ld, const int32_t *count_ptr,
                                                            int rows_host, const int32_t *idmap, int k, int32_t *ids,
                                                            float *vals) {
  __shared__ float sc_v[(kTopkThreads / kWarp) * NS_MAX_TOPK];
  __shared__ int sc_i[(kTopkThreads / kWarp) * NS_MAX_TOPK];
  __shared__ float res_v[NS_MAX_TOPK];
  __shared__ int res_i[NS_MAX_TOPK];
  const int r = blockIdx.x;
  const int m = count_ptr ? *count_ptr : rows_host;
  const float *row = logits + (size_t)r * ld;
  TopList<KMAX> L;
  L.clear();
  for (int j = threadIdx.x; j < m; j += blockDim.x) L.insert(row[j], j);
  block_select<KMAX>(L, k, sc_v, sc_i, res_v, res_i);
  if (threadIdx.x < k) {
    const int j = res_i[threadIdx.x];
    const bool ok = j != kEmptyId;
    ids[(size_t)r * k + threadIdx.x] = ok ? (idmap ? idmap[j] : j) : -1;
    vals[(size_t)r * k + threadIdx.x] = ok ? res_v[threadIdx.x] : -__int_as_float(0x7f800000);
  }
}

}  // namespace

size_t project_smem_bytes() { return (size_t)kProjStages * kStageBytes; }

cudaError_t prepare_project_kernels() {
  return cudaFuncSetAttribute(project_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)project_smem_bytes());
}

cudaError_t launch_project(const ProjArgs &a, int grid, cudaStream_t st) {
  project_kernel<<<grid, kProjThreads, project_smem_bytes(), st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_topk(const float *logits, int ld, const int32_t *count_ptr, int rows_host, const int32_t *idmap,
                        int n, int k, int32_t *ids, float *vals, cudaStream_t st) {
  if (k <= 16) topk_kernel<16><<<n, kTopkThreads, 0, st>>>(logits, ld, count_ptr, rows_host, idmap, k, ids, vals);
  else topk_kernel<32><<<n, kTopkThreads, 0, st>>>(logits, ld, count_ptr, rows_host, idmap, k, ids, vals);
  return cudaGetLastError();
}

}  // namespace ns
