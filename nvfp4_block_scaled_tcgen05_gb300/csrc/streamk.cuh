// Stream-K host and fixup pieces of the BF16 GEMM: the fixup kernel, its
// host-built plan and the share of the tail (the schedule itself is seg_at
// in tcgen05_gemm.cuh).
#pragma once

#include "launch.cuh"

namespace gb300 {

// Stream-K fixup plan, built on the host: for every tail tile whose K
// iterations were divided over several clusters, its position and the
// clusters c0 .. c0+n-1 that hold its partial tiles, in K order.  Cluster
// c0's partial is its last segment (slot 1) unless its iteration range starts
// at the tile's first iteration (slot 0); every later contributor's is its
// first segment (slot 0).  Passed by value (about 3.3 KB of parameters).
constexpr int kSkMaxTail = 256;
struct StreamKPlan {
  uint32_t mb[kSkMaxTail], nb[kSkMaxTail];  // output tile (M block, N block)
  uint16_t c0[kSkMaxTail], n[kSkMaxTail];   // first contributing cluster, count (>= 2)
  uint8_t slot0[kSkMaxTail];                // workspace slot of c0's partial
  int tiles;                                // split tiles listed
};

// Stream-K fixup (BF16 GEMM): a split tile is the FP32 sum of its partial
// tiles taken in K order, rounded once to BF16 (tiles computed by one
// cluster were stored by it).  Grid (split tiles, TILE_M / 4): 4 rows x 256 columns per CTA, 4
// consecutive columns per thread, the loads of up to eight partials in flight
// ahead of the ordered adds.  Launched as a programmatic dependent of the
// GEMM: it is scheduled while the GEMM's last tiles run and waits for the
// GEMM's completion in griddep_wait().
constexpr int kFixupBatch = 8;
template <class Cfg>
__global__ void __launch_bounds__(256)
    streamk_fixup_kernel(const __grid_constant__ StreamKPlan plan, const GemmParams p,
                         const float* __restrict__ ws) {
  static_assert(Cfg::BN == 256, "64 threads x 4 columns cover a row");
  const int t = int(blockIdx.x);
  const int c0 = plan.c0[t], n = plan.n[t];
  const int r = int(blockIdx.y) * 4 + int(threadIdx.x) / 64;
  const int col = (int(threadIdx.x) % 64) * 4;
  const int grow = int(plan.mb[t]) * Cfg::TILE_M + r, gcol = int(plan.nb[t]) * Cfg::BN + col;
  ptx::griddep_wait();
  if (grow >= p.M || gcol >= p.N) return;
  constexpr size_t kSlot = size_t(Cfg::TILE_M) * Cfg::BN;
  const float* base = ws + size_t(r) * Cfg::BN + col;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = 0; i < n; i += kFixupBatch) {
    float4 v[kFixupBatch];
#pragma unroll
    for (int u = 0; u < kFixupBatch; ++u) {
      const int k = i + u;  // contributor c0 + k
      const size_t slot = size_t(c0 + k) * 2 + ((k == 0) ? plan.slot0[t] : 0);
      if (k < n) v[u] = *reinterpret_cast<const float4*>(base + slot * kSlot);
    }
#pragma unroll
    for (int u = 0; u < kFixupBatch; ++u) {
      const int k = i + u;
      if (k >= n) break;
      if (k == 0) {
        acc = v[u];
      } else {
        acc.x += v[u].x;
        acc.y += v[u].y;
        acc.z += v[u].z;
        acc.w += v[u].w;
      }
    }
  }
  uint2 o;
  o.x = pack_bf16x2(__float_as_uint(acc.x), __float_as_uint(acc.y));
  o.y = pack_bf16x2(__float_as_uint(acc.z), __float_as_uint(acc.w));
  *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.c_ptr) + size_t(grow) * p.N + gcol) = o;
}

// The fixup plan of a stream-K launch (p.sk = P clusters sharing the tail of
// T = (tiles mod C) * kbt iterations, P <= T): cluster c takes iterations
// [T*c/P, T*(c+1)/P), so the owner of iteration x is ceil((x+1)*P/T) - 1.
template <class Cfg>
void build_streamk_plan(const GemmParams& p, int C, StreamKPlan& plan) {
  const int P = p.sk;
  const int dp_rounds = p.total_tiles / C;
  const int tail = p.total_tiles - dp_rounds * C;
  const long long kbt = p.num_k_blocks;
  const long long T = (long long)tail * kbt;
  plan.tiles = 0;
  for (int t = 0; t < tail; ++t) {
    const long long ts = t * kbt, te = ts + kbt;
    const int c0 = int(((ts + 1) * P + T - 1) / T - 1);
    const int c1 = int((te * P + T - 1) / T - 1);
    if (c1 == c0) continue;
    int l, mb, nb;
    decode_tile<Cfg>(dp_rounds * C + t, p, l, mb, nb);
    const int i = plan.tiles++;
    plan.mb[i] = uint32_t(mb);
    plan.nb[i] = uint32_t(nb);
    plan.c0[i] = uint16_t(c0);
    plan.n[i] = uint16_t(c1 - c0 + 1);
    plan.slot0[i] = uint8_t((T * c0 / P == ts) ? 0 : 1);
  }
}


// Among P = 1..C, the P that minimises ceil(T / P) K iterations on the
// critical path plus 0.1 iteration for each partial tile written and summed
// (T / P + tail of them), the ratio measured on the 5120 x 2048 x {2048,
// 11008} BF16 GEMMs.
inline int streamk_min_cost_share(long long T, int tail, int C) {
  int best = C;
  double best_cost = 1e300;
  for (int P = 1; P <= C; ++P) {
    const double cost = double((T + P - 1) / P) + 0.1 * double(P + tail);
    if (cost < best_cost) {
      best_cost = cost;
      best = P;
    }
  }
  return best;
}

// The fixup grid (split tiles, TILE_M / 4), launched as a programmatic
// dependent of the GEMM.
template <class Cfg>
int launch_streamk_fixup(const StreamKPlan& plan, const GemmParams& p, const float* ws,
                         cudaStream_t stream) {
  static_assert(sizeof(StreamKPlan) + sizeof(GemmParams) + sizeof(void*) <= 4096,
                "kernel parameters fit the classic 4 KB limit");
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(plan.tiles, Cfg::TILE_M / 4);
  cfg.blockDim = dim3(256);
  if (cudaLaunchKernelEx(&cfg, streamk_fixup_kernel<Cfg>, plan, p, ws) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

}  // namespace gb300
