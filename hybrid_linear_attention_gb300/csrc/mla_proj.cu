// mla_proj.cu -- the absorbed gated-MLA decode's two projections on the tensor cores.
//
// "Ling-3.1-flash: Grouped Routing and Two Different MLA Caches", section "Why weight
// absorption keeps the same attention function": the key up-projection W_K,i moves into the
// query, q~_i = W_K,i^T q_i^N (512 wide), and the value up-projection W_V,i comes after the
// latent-weighted sum, o_i = W_V,i z_i, scaled by the head's sigmoid gate.  Across the
// sequences of a decode batch both are, per head, dense products (a batch of query rows
// against one 128 x 512 weight), so each runs as tcgen05 MMAs on 128-sequence tiles.
//
//   mla_absorb_tc_kernel   CTA (latent half, head, 128 sequences): D[b][l] = sum_n q^N[b][n]
//                          W_K[n][l], M = 128 sequences, N = 256 latent channels, K = 128;
//                          A = q^N K-major, B = W_K read MN-major straight from its [n][l]
//                          layout (both by TMA, 128-byte swizzle); bf16 in, fp32 in tensor
//                          memory, bf16 out into q_cat, with q^R copied behind it.
//   mla_up_gate_tc_kernel  CTA (head, 128 sequences): D[b][v] = sum_l z[b][l] W_V[v][l],
//                          M = 128 sequences, N = 128, K = 512 in stages of 64; z (fp32)
//                          is split on the CUDA cores into bf16 hi + lo (two products, the
//                          sum good to ~2^-17 relative), W_V K-major by TMA; the epilogue
//                          scales each row by sigmoid(gate) and writes bf16.
#include <atomic>
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_tc_ptx.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int PH = 64, PL = 512, PR = 64, PK = PL + PR, PN = 128, PV = 128;
constexpr int PB = 128;            // sequences per CTA (the MMA's M)
constexpr int PT = 128;            // threads per CTA: one TMEM lane (sequence row) each
constexpr long kProjWaitLimit = 1L << 24;

// rows of a batch box: a tensor-map box may not be larger than the tensor, so a batch of fewer
// than 128 sequences is loaded whole (the MMA rows past it read whatever the buffer holds and
// are never stored)
__host__ __device__ constexpr uint32_t box_rows(int B) { return B < PB ? (uint32_t)B : (uint32_t)PB; }

__device__ __forceinline__ bool proj_wait(uint32_t bar, uint32_t parity) {
#pragma unroll 1
  for (long it = 0; it < kProjWaitLimit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

struct ProjMaps {
  CUtensorMap a, w, z;
};

// ---- absorption ---------------------------------------------------------------------------
constexpr uint32_t AB_A = 0;        // q^N: 2 panels [128 rows][64 ch] bf16, 16 KB each
constexpr uint32_t AB_W = 32768;    // W_K half: 4 atoms [128 n][64 l] bf16, 16 KB each
constexpr uint32_t AB_SMEM = 32768 + 65536 + 1024;

__global__ void __launch_bounds__(PT, 1)
    mla_absorb_tc_kernel(const MlaArgs a, const __grid_constant__ ProjMaps maps) {
  extern __shared__ uint8_t praw[];
  __shared__ __align__(8) uint64_t s_bar[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_fail;
  const uint32_t raw = smem_u32(praw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  const int half = blockIdx.x, h = blockIdx.y, b0 = blockIdx.z * PB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(smem_u32(&s_bar[0]), 1);
    mbar_init(smem_u32(&s_bar[1]), 1);
    mbar_fence_init();
    s_fail = 0;
  }
  if (warp == 0) tmem_alloc(smem_u32(&s_tmem), 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = s_tmem;
  if (tid == 0) {
    const uint32_t ld = smem_u32(&s_bar[0]), mm = smem_u32(&s_bar[1]);
    mbar_expect_tx(ld, 2u * 128u * box_rows(a.B) + 65536u);
    for (int p = 0; p < 2; ++p) tma_load_3d(sb + AB_A + 16384u * p, &maps.a, 64 * p, h, b0, ld);
    for (int at = 0; at < 4; ++at)
      tma_load_3d(sb + AB_W + 16384u * at, &maps.w, 256 * half + 64 * at, 0, h, ld);
    if (proj_wait(ld, 0)) {
      tc_fence_after();
      constexpr uint32_t ID = idesc(1, 128, 256, 0, 1);  // bf16, A K-major, B MN-major
      for (int ks = 0; ks < PN / 16; ++ks) {
        const uint64_t ad = sdesc_sw128(sb + AB_A + (ks >> 2) * 16384u + (ks & 3) * 32u, 16, 1024);
        const uint64_t bd = sdesc_sw128(sb + AB_W + (uint32_t)ks * 2048u, 16384, 1024);
        mma_bf16_ss(tm, ad, bd, ID, ks > 0);
      }
      mma_commit(mm);
      if (!proj_wait(mm, 0)) s_fail = 1;
    } else {
      s_fail = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int b = b0 + 32 * warp + lane;  // this thread's TMEM lane = sequence row
  if (!s_fail) {
    bf16 *row = reinterpret_cast<bf16 *>(a.q_cat) + ((size_t)b * PH + h) * PK + 256 * half;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      float v[32];
      tmem_ld32(tm + ((uint32_t)(32 * warp) << 16) + 32u * c, v);
      tmem_wait_ld();
      if (b < a.B) {
        uint32_t w[16];
#pragma unroll
        for (int y = 0; y < 16; ++y) {
          const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * y]));
          const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * y + 1]));
          w[y] = lo | (hi << 16);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(row + 32 * c);
#pragma unroll
        for (int y = 0; y < 4; ++y) dst[y] = make_uint4(w[4 * y], w[4 * y + 1], w[4 * y + 2], w[4 * y + 3]);
      }
    }
    if (half == 1 && b < a.B) {  // q^R behind the absorbed part
      const uint4 *src =
          reinterpret_cast<const uint4 *>(reinterpret_cast<const bf16 *>(a.q_rope) + ((size_t)b * PH + h) * PR);
      uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<bf16 *>(a.q_cat) + ((size_t)b * PH + h) * PK + PL);
#pragma unroll
      for (int y = 0; y < PR / 8; ++y) dst[y] = src[y];
    }
  } else if (tid == 0 && a.err) {
    atomicOr(a.err, ERR_MBAR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, 256);
}

// ---- value up-projection and gate ----------------------------------------------------------
// per stage s (latent channels 64 s .. 64 s + 63), four stages in flight: z raw fp32 (two
// boxes of [128 rows][32], 16 KB each), W_V [128 v][64 l] bf16 (16 KB).  Each thread turns its
// own row of z into bf16 hi | lo in place: hi over the first box's row, lo over the second's
// ([128][64] bf16 each, the same 128-byte pitch and swizzle)
constexpr uint32_t UG_STAGE = 32768 + 16384;
constexpr uint32_t UG_Z = 0, UG_W = 32768, UG_HI = 0, UG_LO = 16384;
constexpr int UG_NB = 4;  // stage buffers
constexpr uint32_t UG_SMEM = UG_NB * UG_STAGE + 1024;
constexpr int UG_NS = PL / 64;

__global__ void __launch_bounds__(PT, 1)
    mla_up_gate_tc_kernel(const MlaArgs a, const __grid_constant__ ProjMaps maps) {
  extern __shared__ uint8_t praw[];
  __shared__ __align__(8) uint64_t s_bar[2 * UG_NB];  // loads landed, products done (by buffer)
  __shared__ uint32_t s_tmem;
  __shared__ int s_fail;
  const uint32_t raw = smem_u32(praw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t *sm = praw + pad;
  const uint32_t sb = raw + pad;
  const int h = blockIdx.x, b0 = blockIdx.y * PB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < 2 * UG_NB; ++i) mbar_init(smem_u32(&s_bar[i]), 1);
    mbar_fence_init();
    s_fail = 0;
  }
  if (warp == 0) tmem_alloc(smem_u32(&s_tmem), 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = s_tmem;
  auto ld_bar = [&](int j) { return smem_u32(&s_bar[j]); };
  auto mm_bar = [&](int j) { return smem_u32(&s_bar[UG_NB + j]); };
  auto load = [&](int s) {  // thread 0: stage s into buffer s % UG_NB
    const int j = s % UG_NB;
    const uint32_t base = sb + (uint32_t)j * UG_STAGE;
    mbar_expect_tx(ld_bar(j), 2u * 128u * box_rows(a.B) + 16384u);
    tma_load_3d(base + UG_Z, &maps.z, 64 * s, h, b0, ld_bar(j));
    tma_load_3d(base + UG_Z + 16384, &maps.z, 64 * s + 32, h, b0, ld_bar(j));
    tma_load_3d(base + UG_W, &maps.w, 64 * s, 0, h, ld_bar(j));
  };
  if (tid == 0)
    for (int s = 0; s < UG_NB && s < UG_NS; ++s) load(s);
  constexpr uint32_t ID = idesc(1, 128, 128, 0, 0);  // bf16, both K-major
  bool ok = true;
#pragma unroll 1
  for (int s = 0; s < UG_NS && ok; ++s) {
    const int j = s % UG_NB;
    uint8_t *stg = sm + (uint32_t)j * UG_STAGE;
    if (!proj_wait(ld_bar(j), (uint32_t)((s / UG_NB) & 1))) s_fail = 1;
    // row tid: its 64 fp32 values (two swizzled 128-byte rows) -> bf16 hi | lo, K-major
    // [128 rows][64] with the same 128-byte swizzle, over the same two rows: every value of
    // the row is read before the first write
    float xa[2][4][8];
#pragma unroll
    for (int box = 0; box < 2; ++box) {
      const uint8_t *zr = stg + UG_Z + 16384u * box + (uint32_t)tid * 128u;
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // 16-byte pieces of 8 fp32 = pieces 2q, 2q + 1
        const float4 x0 = *reinterpret_cast<const float4 *>(zr + (((2 * q) ^ (tid & 7)) << 4));
        const float4 x1 = *reinterpret_cast<const float4 *>(zr + (((2 * q + 1) ^ (tid & 7)) << 4));
        xa[box][q][0] = x0.x, xa[box][q][1] = x0.y, xa[box][q][2] = x0.z, xa[box][q][3] = x0.w;
        xa[box][q][4] = x1.x, xa[box][q][5] = x1.y, xa[box][q][6] = x1.z, xa[box][q][7] = x1.w;
      }
    }
#pragma unroll
    for (int box = 0; box < 2; ++box) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float(&xs)[8] = xa[box][q];
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const __nv_bfloat16 h0 = __float2bfloat16_rn(xs[2 * y]), h1 = __float2bfloat16_rn(xs[2 * y + 1]);
          const __nv_bfloat16 l0 = __float2bfloat16_rn(xs[2 * y] - __bfloat162float(h0));
          const __nv_bfloat16 l1 = __float2bfloat16_rn(xs[2 * y + 1] - __bfloat162float(h1));
          hw[y] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
          lw[y] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
        }
        // channel 32 box + 8 q .. + 7 of the stage = bf16 piece 4 box + q of the 128-byte row
        const uint32_t off = (uint32_t)tid * 128u + ((uint32_t)((4 * box + q) ^ (tid & 7)) << 4);
        *reinterpret_cast<uint4 *>(stg + UG_HI + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4 *>(stg + UG_LO + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (s_fail) {
      ok = false;
      break;
    }
    if (tid == 0) {
      const uint32_t base = sb + (uint32_t)j * UG_STAGE;
      for (int term = 0; term < 2; ++term)
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ad = sdesc_sw128(base + (term ? UG_LO : UG_HI) + (uint32_t)ks * 32u, 16, 1024);
          const uint64_t bd = sdesc_sw128(base + UG_W + (uint32_t)ks * 32u, 16, 1024);
          mma_bf16_ss(tm, ad, bd, ID, (s | term | ks) != 0);
        }
      mma_commit(mm_bar(j));
      if (s + UG_NB < UG_NS) {  // buffer j is free once these products have read it
        if (!proj_wait(mm_bar(j), (uint32_t)((s / UG_NB) & 1))) s_fail = 1;
        else load(s + UG_NB);
      }
    }
  }
  // the last products (stages UG_NS - UG_NB .. UG_NS - 1, one per buffer)
  if (ok && tid == 0)
    for (int s = UG_NS - UG_NB; s < UG_NS; ++s)
      if (!proj_wait(mm_bar(s % UG_NB), (uint32_t)((s / UG_NB) & 1))) s_fail = 1;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int b = b0 + 32 * warp + lane;
  if (!s_fail) {
    const float gl = b < a.B ? __bfloat162float(reinterpret_cast<const bf16 *>(a.gate)[(size_t)b * PH + h]) : 0.f;
    const float gs = sigmoidf_(gl);
    bf16 *row = reinterpret_cast<bf16 *>(a.out) + ((size_t)b * PH + h) * PV;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      float v[32];
      tmem_ld32(tm + ((uint32_t)(32 * warp) << 16) + 32u * c, v);
      tmem_wait_ld();
      if (b < a.B) {
        uint32_t w[16];
#pragma unroll
        for (int y = 0; y < 16; ++y) {
          const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * y] * gs));
          const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * y + 1] * gs));
          w[y] = lo | (hi << 16);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(row + 32 * c);
#pragma unroll
        for (int y = 0; y < 4; ++y) dst[y] = make_uint4(w[4 * y], w[4 * y + 1], w[4 * y + 2], w[4 * y + 3]);
      }
    }
  } else if (tid == 0) {
    // a bounded wait ran out: let the copies and products in flight land (bounded), then report
    for (int i = 0; i < 2 * UG_NB; ++i) proj_wait(smem_u32(&s_bar[i]), 0), proj_wait(smem_u32(&s_bar[i]), 1);
    if (a.err) atomicOr(a.err, ERR_MBAR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, 128);
}

bool proj_map(CUtensorMap *m, const void *ptr, bool f32, uint64_t d0, uint64_t d1, uint64_t d2,
              uint32_t b0, uint32_t b1, uint32_t b2) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  const int es = f32 ? 4 : 2;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * es, d0 * d1 * es};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t el[3] = {1, 1, 1};
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void *>(ptr), dims, strides, box, el, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// the dynamic shared-memory opt-in of one kernel, once per device (each kernel passes its own
// flags: both kernels have the same signature, so a per-type cache would be shared)
template <typename K>
cudaError_t set_smem(K kernel, uint32_t bytes, std::atomic<bool> (&done)[64]) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !done[dev].load()) {  // idempotent if two threads race here
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    done[dev].store(true);
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_mla_absorb(const MlaArgs &a, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  ProjMaps maps;
  std::memset(&maps, 0, sizeof maps);
  // q^N [B][64][128]: boxes of 64 channels x 1 head x 128 sequences (the last box of a batch
  // reads zeros past B; a batch under 128 sequences is one box of B rows);
  // W_K [64][128][512]: boxes of 64 latent x 128 n x 1 head
  if (!proj_map(&maps.a, a.q_nope, false, PN, PH, (uint64_t)a.B, 64, 1, box_rows(a.B)) ||
      !proj_map(&maps.w, a.w_uk, false, PL, PN, PH, 64, PN, 1))
    return cudaErrorInvalidValue;
  static std::atomic<bool> attr_set[64];
  cudaError_t e = set_smem(mla_absorb_tc_kernel, AB_SMEM, attr_set);
  if (e != cudaSuccess) return e;
  mla_absorb_tc_kernel<<<dim3(2, PH, (a.B + PB - 1) / PB), PT, AB_SMEM, s>>>(a, maps);
  return cudaGetLastError();
}

cudaError_t launch_mla_up_gate(const MlaArgs &a, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  ProjMaps maps;
  std::memset(&maps, 0, sizeof maps);
  // z [B][64][512] fp32: boxes of 32 channels x 1 head x 128 sequences; W_V [64][128][512]:
  // boxes of 64 latent x 128 v x 1 head (K-major)
  if (!proj_map(&maps.z, a.z, true, PL, PH, (uint64_t)a.B, 32, 1, box_rows(a.B)) ||
      !proj_map(&maps.w, a.w_uv, false, PL, PV, PH, 64, PV, 1))
    return cudaErrorInvalidValue;
  static std::atomic<bool> attr_set[64];
  cudaError_t e = set_smem(mla_up_gate_tc_kernel, UG_SMEM, attr_set);
  if (e != cudaSuccess) return e;
  mla_up_gate_tc_kernel<<<dim3(PH, (a.B + PB - 1) / PB), PT, UG_SMEM, s>>>(a, maps);
  return cudaGetLastError();
}

}  // namespace kda
