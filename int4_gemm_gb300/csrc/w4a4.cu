// W4A4 GEMM on the GB300 FP4 tensor cores: C = A_hat . B_hat^T with E2M1
// operands and per-16 E4M3 (NVFP4) or per-32 E8M0 (MXFP4) block scales
// ("Low-bit inference for very large MoE", section "Kernels on different
// hardware": activations quantized to FP4 too, both operands enter the FP4
// tensor cores; "Quantization in deployment", "Fake quantization" for the
// formats).  Also the grouped routed-MoE variant (same section: one low-bit
// weight matrix per expert, grouped by routing).
//
// Structure (one persistent CTA per SM; on large problems the CTAs work in
// pairs, see P2 below):
//   warp 0     code producer: TMA tiles of packed codes (128-byte swizzle)
//              into a 4- or 5-stage shared-memory ring.
//   warp 10    scale producer: bulk copies of the stage's scale tiles into the
//              same stage (its own arrival on the stage's barrier), so the
//              two producers issue their copies in parallel (prefill GEMM
//              656 -> 634 us against one producer issuing all of them).
//   warp 1     allocates TMEM; one lane issues tcgen05.mma ... block_scale,
//              128xBNTx64 per instruction, FP32 accumulation in TMEM.
//   warps 2-5  epilogue: tcgen05.ld of the 128x256 FP32 accumulator, times
//              gA * gB (NVFP4), rounded to bf16 (or kept FP32), stored.
//   warps 6-9  scale writers: each stage's scale tiles go from shared memory
//              to TMEM through registers (tcgen05.st, one warp per TMEM lane
//              quarter).  Unlike tcgen05.cp these stores do not queue behind
//              the MMAs in the tensor pipe, so the MMA thread issues nothing
//              but MMAs.
// P2 (pairs): a cluster of 2 CTAs computes one 256x256 tile with the 2-SM MMA
// (tcgen05 ... cta_group::2, 256x256x64 per instruction): each CTA holds its
// 128 rows of A and its 128-row half of B in shared memory, and all 256 rows
// of B's scales with its own A scales in its TMEM; the even CTA issues the
// MMAs and each CTA's accumulator receives its 128 rows.  Each SM thus
// receives half of the B tile per stage.  The odd CTA's scale writers and
// epilogue warps report to the even CTA's barriers.
// QA (MXFP4 with a raw A, gemm_w4a4_mxfp4_fused): the GEMM quantizes its
// activations itself, in a prologue: warps 1-9 of every CTA encode that CTA's
// share of A's 32-element blocks into the workspace (codes and
// tensor-core-layout scales) and the CTA counts itself in a grid-wide gate;
// meanwhile the producers already stream the first stages' B tiles and issue
// the A copies once every CTA has passed the gate.  Each element is encoded
// once; one launch replaces quantizer + GEMM.  The grid is never larger than
// what is resident at once, so the gate is always reached; its wait is
// bounded like every other.  The gate is two counters (arrivals, then
// departures of the two waiting producers of every CTA); the last waiter to
// leave sets both back to zero, so a workspace that starts at zero stays
// ready for the next launch without a reset of its own.
// Every wait is bounded: on timeout the CTA latches Q4_ERR_TIMEOUT, drains
// its own copies and MMAs, frees TMEM and exits.
#include "common.cuh"
#include "internal.h"
#include "quant_device.cuh"

#include <algorithm>

namespace q4 {
namespace {

constexpr int BM = 128, BN = 256, BK = 256;   // BK in elements (128 bytes of codes); BN: widest N tile
constexpr int kMaxStages = 5;
constexpr int kThreads = 192;          // code producer, MMA, 4 epilogue warps
constexpr int kWriterThreads = 128;    // 4 scale-writer warps
constexpr int kWriterWarp0 = (kThreads + kWriterThreads) / 32 - 4;  // warps 6-9
template <bool GROUPED>
constexpr int block_threads() { return kThreads + kWriterThreads + 32; }  // + the scale producer warp
constexpr uint32_t kABytes = BM * BK / 2;     // 16 KiB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfColsPerStage = 48;      // 16 (A) + 32 (B: two 128-row chunks)
constexpr int kMaxExperts = 1024;

__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t local_addr, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(ra)
               : "memory");
  return v;
}

// Stage: [A codes | B codes (all BN rows, or this CTA's half in pairs) |
// A scales (128 rows) | B scales (256 rows)]
// BNT: N tile width (256; 128 for split-K on few output tiles).
template <bool NV, bool P2 = false, int BNT = BN>
struct Cfg {
  static constexpr uint32_t kBBytes = BNT * BK / 2;
  static constexpr uint32_t kAccCols = BNT;   // FP32 accumulator columns
  static constexpr int kPartStride = BNT + 4;  // FP32 partial tile row stride (split-K), padded against bank conflicts
  static constexpr int kStages = P2 ? 5 : (BNT == 128 ? 5 : 4);
  static constexpr uint32_t kSfaBytes = NV ? 2048u : 1024u;  // 128 rows x (16 | 8) scales
  static constexpr uint32_t kSfbBytes = 2 * kSfaBytes;        // 256 rows
  static constexpr uint32_t kBLoad = P2 ? kBBytes / 2 : kBBytes;
  static constexpr uint32_t kSfaOff = kABytes + kBLoad;
  static constexpr uint32_t kSfbOff = kSfaOff + kSfaBytes;
  static constexpr uint32_t kStageBytes = kSfbOff + kSfbBytes;
  static constexpr uint32_t kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
  static constexpr uint32_t kSfChunks = NV ? 4u : 2u;  // 512-byte chunks per 128 rows per stage
};
static_assert(Cfg<true>::kStageBytes % 1024 == 0 && Cfg<false>::kStageBytes % 1024 == 0, "");
static_assert(Cfg<true, true>::kStageBytes % 1024 == 0 && Cfg<false, true>::kStageBytes % 1024 == 0, "");
static_assert(Cfg<true>::kSmemBytes <= 232448 && Cfg<true, true>::kSmemBytes <= 232448, "shared memory");
static_assert(BN + kMaxStages * kSfColsPerStage <= kTmemCols, "TMEM columns");
static_assert(Cfg<true, false, 128>::kSmemBytes <= 232448 && Cfg<false, false, 128>::kStageBytes % 1024 == 0, "");

struct Smem {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t sf_full[kMaxStages];  // the stage's scales are in TMEM
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

struct TileInfo {
  int m_row0;    // first output row of the tile
  int m_end;     // output rows < m_end are valid
  int n0;        // first output column
  int sf_block;  // A scale row-block (dense: m tile; grouped: tile-row)
  int e;         // expert (grouped) or 0
  bool ok;
};

struct Params {
  int64_t M, N, K;
  const uint8_t* a_sf;    // MMA layout
  const uint8_t* b_sf;    // MMA layout (grouped: E consecutive tensors)
  int64_t b_sf_expert_bytes;
  const float* a_g;
  const float* b_g;       // grouped: [E]
  void* C;
  int c_dtype;
  int num_m, num_n;       // dense tile counts
  int bn;                 // N tile width (the kernel's BNT)
  // grouped
  const int32_t* offsets;
  const int32_t* sched;
  int E;
  // activations quantized in the prologue (QA): raw A, its dtype, where its
  // codes and tensor-core-layout scales go, and the gate the CTAs count into
  const void* a_raw;
  int a_dtype;
  uint8_t* a_codes_w;
  uint8_t* a_sf_w;
  unsigned* gate;
  // split-K: [tile][rank][BNT / 4][BM] float4 partial sums in global memory
  // (they meet in L2); nullptr: through distributed shared memory
  float4* part_g;
  KernelCtl ctl;
};

__device__ __forceinline__ void bar_sync_n(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Waits (bounded) until every CTA of the grid has counted itself in gate[0],
// then orders the copies (async proxy) this thread issues next after the
// other CTAs' generic-proxy stores it has now seen, and counts itself out in
// gate[1]; the last of the grid's `waiters` to leave resets both counters
// (nobody reads them any more in this launch, and the next launch on the
// workspace reads them only after this one has completed).
__device__ __forceinline__ bool wait_gate(unsigned* gate, unsigned target, unsigned waiters,
                                          const KernelCtl& ctl, volatile int* abort_flag) {
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(gate) : "memory");
    if (v >= target) break;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > ctl.wait_ns) {
      latch_status(ctl.status, Q4_ERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
    __nanosleep(64);
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  if (atomicAdd(gate + 1, 1u) == waiters - 1) {
    *reinterpret_cast<volatile unsigned*>(gate) = 0u;
    *reinterpret_cast<volatile unsigned*>(gate + 1) = 0u;
  }
  return true;
}

// The QA prologue: this CTA's blocks [c B / G, (c + 1) B / G) of the M x K/32
// MXFP4 blocks of A, one thread per 16 elements (a lane pair per block), by
// threads t = 0 .. nthr - 1 (whole warps).  A CTA's share is small (a few
// tens of KB), so its time is load latency: each thread first issues the
// loads of up to kPU units, then encodes them.
template <typename T>
__device__ void mxfp4_prologue(const Params& p, int t, int nthr) {
  constexpr int kPU = 4;
  const T* x = static_cast<const T*>(p.a_raw);
  const uint32_t nblk = (uint32_t)(p.K / 16);  // units per row
  const int64_t nsf4 = (p.K / 32 + 3) / 4;
  const int64_t B = p.M * (p.K / 32);
  const int64_t u_lo = 2 * ((int64_t)blockIdx.x * B / gridDim.x);
  const int64_t u_hi = 2 * ((int64_t)(blockIdx.x + 1) * B / gridDim.x);
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)kPU * nthr;
  for (int64_t c0 = u_lo + (t & ~31); c0 < u_hi; c0 += stride) {  // warp-uniform trip count
    Raw16<T> raw[kPU];
#pragma unroll
    for (int i = 0; i < kPU; ++i) {
      const int64_t u = c0 + (int64_t)i * nthr + lane;
      if (u < u_hi) load_raw16<T>(x, u * 16, raw[i]);
    }
#pragma unroll
    for (int i = 0; i < kPU; ++i) {
      const int64_t u = c0 + (int64_t)i * nthr + lane;
      const bool live = u < u_hi;
      float v[16];
      float amax = 0.f;
      if (live) {
        unpack16<T>(raw[i], v);
#pragma unroll
        for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));  // the block's other half
      if (!live) continue;
      int e;
      reinterpret_cast<uint2*>(p.a_codes_w)[u] = mxfp4_encode16(v, amax, false, e);
      if ((u & 1) == 0) {
        const uint32_t row = (uint32_t)u / nblk;
        const uint32_t blk = ((uint32_t)u - row * nblk) >> 1;
        p.a_sf_w[mma_scale_offset(row, blk, nsf4)] = (uint8_t)(e + 127);
      }
    }
  }
}

// Dense tiles for CM CTAs stacked along M (CM = 2: a CTA pair sharing one
// 256-wide N tile): cluster tile t -> (m group, n) in bands of 64 M tiles
// (8192 rows: A and its scales, up to 38 MB, stay in L2), so B streams from
// DRAM once per band (bands of 16 M tiles read the prefill B four times and
// were 3% slower); CTA rank r takes M tile group * CM + r.
template <int CM>
__device__ __forceinline__ TileInfo dense_tile(const Params& p, int t, int crank) {
  constexpr int GMG = 64 / CM;  // m groups per band
  const int num_mg = (p.num_m + CM - 1) / CM;
  TileInfo ti;
  const int band_tiles = GMG * p.num_n;
  const int band = t / band_tiles, r = t % band_tiles;
  const int gm = min(GMG, num_mg - band * GMG);
  const int mg = band * GMG + r % gm, n = r / gm;
  const int m = mg * CM + crank;
  ti.m_row0 = m * BM;
  ti.m_end = (int)p.M;
  ti.n0 = n * p.bn;
  ti.sf_block = m;
  ti.e = 0;
  ti.ok = true;
  return ti;
}

// Grouped tiles: tile-row tr (expert-major, one per 128 routed rows of an
// expert) x n tile; n varies fastest so an expert's weights are reused from
// L2 by all of its tile-rows.
__device__ __forceinline__ TileInfo grouped_tile(const Params& p, const int* sched, int t) {
  TileInfo ti;
  const int tr = t / p.num_n, n = t % p.num_n;
  int e = 0;
  while (e + 1 < p.E && sched[e + 1] <= tr) ++e;
  ti.e = e;
  ti.m_row0 = __ldg(p.offsets + e) + (tr - sched[e]) * BM;
  ti.m_end = __ldg(p.offsets + e + 1);
  ti.n0 = n * p.bn;
  ti.sf_block = tr;
  ti.ok = ti.m_row0 < ti.m_end;
  return ti;
}


// KS > 1: split-K -- a cluster of KS CTAs owns one output tile, each CTA a
// slice of the K blocks; the FP32 partial tiles are reduced through
// distributed shared memory in rank order (deterministic).
template <bool NV, bool GROUPED, int KS = 1, bool P2 = false, int BNT = BN, bool QA = false>
__global__ void __launch_bounds__(block_threads<GROUPED>(), 1)
    fp4_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b, const Params p) {
  using C_ = Cfg<NV, P2, BNT>;
  static_assert(BNT == BN || (BNT == 128 && !P2), "N tile: 256, or 128 without pairs");
  constexpr uint32_t kAccCols = C_::kAccCols;
  constexpr int kPartStride = C_::kPartStride;
  constexpr int kStages = C_::kStages;
  extern __shared__ uint8_t smem_raw[];
  pdl_wait();  // operands, scales and the schedule may come from the previous kernel
  // 1024-byte alignment for the 128-byte swizzle atoms
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Smem* sm = reinterpret_cast<Smem*>(smem + kStages * C_::kStageBytes);
  __shared__ int s_sched[GROUPED ? kMaxExperts + 1 : 1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  static_assert(!P2 || (KS == 1 && !GROUPED), "");
  static_assert(KS == 1 || !GROUPED, "");
  static_assert(!QA || (!NV && !GROUPED), "the prologue quantizes dense MXFP4 activations");
  constexpr int TM = P2 ? 2 : 1;                           // CTAs along M per tile
  constexpr int CL = TM * KS;                              // CTAs per cluster
  const int crank = P2 ? (int)cluster_ctarank() : 0;      // rank in the pair
  const int krank = KS > 1 ? (int)cluster_ctarank() : 0;  // rank along K (split-K)
  const bool leader = crank == 0;                          // issues the pair's MMAs
  const int cid = blockIdx.x / CL, ncl = gridDim.x / CL;   // cluster index and count
  const int nkb_all = (int)(p.K / BK);
  const int kbs = (nkb_all + KS - 1) / KS;
  const int kb_begin = min(nkb_all, krank * kbs), kb_end = min(nkb_all, kb_begin + kbs);

  int total_tiles;
  if constexpr (GROUPED) {
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s_sched[i] = __ldg(p.sched + i);
    __syncthreads();
    total_tiles = s_sched[p.E] * p.num_n;
  } else {
    total_tiles = ((p.num_m + TM - 1) / TM) * p.num_n;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm->full[s]), 2);  // code producer + scale producer
      mbar_init(smem_u32(&sm->empty[s]), 1);
      mbar_init(smem_u32(&sm->sf_full[s]), P2 ? 8 : 4);  // one arrival per scale-writer warp
    }
    mbar_init(smem_u32(&sm->acc_full), 1);
    mbar_init(smem_u32(&sm->acc_empty), P2 ? 8 : 4);  // one arrival per epilogue warp
    mbar_init(smem_u32(&sm->mma_done), 1);
    sm->abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
  }
  if (warp == 1) {
    if constexpr (P2) {
      tmem_alloc_pair(smem_u32(&sm->tmem_base), kTmemCols);  // both CTAs of the pair, same columns
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&sm->tmem_base), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CL > 1) cluster_barrier_sync();  // peers' barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  volatile int* abort_flag = &sm->abort;

  // QA: the prologue runs after the setup, while the producers already
  // stream B (issuing B first measured faster than quantizing first)
  if constexpr (QA) {
    if (warp >= 1 && warp < kWriterWarp0 + 4) {  // warps 1-9: the prologue
      constexpr int kPro = (kWriterWarp0 + 4 - 1) * 32;
      const int t = threadIdx.x - 32;
      if (p.a_dtype == Q4_F32) mxfp4_prologue<float>(p, t, kPro);
      else if (p.a_dtype == Q4_F16) mxfp4_prologue<__half>(p, t, kPro);
      else mxfp4_prologue<__nv_bfloat16>(p, t, kPro);
      // the codes and scales are read next by other CTAs' copies (async
      // proxy); one release after the CTA barrier publishes all its threads'
      // stores with the arrival
      asm volatile("fence.proxy.async.global;" ::: "memory");
      bar_sync_n(2, kPro);
      if (t == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.gate) : "memory");
    }
  }

  // arrive on the pair leader's copy of a barrier (this CTA's own when not paired)
  auto arrive_leader = [&](uint64_t* bar) {
    if constexpr (P2) mbar_arrive_cluster(mapa_shared(smem_u32(bar), 0));
    else mbar_arrive(smem_u32(bar));
  };
  auto tile_at = [&](int t) -> TileInfo {
    if constexpr (GROUPED) return grouped_tile(p, s_sched, t);
    else return dense_tile<TM>(p, t, crank);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t stage = 0, phase = 0;
    int issued[kStages];
    uint32_t issued_phase[kStages];
    for (int s = 0; s < kStages; ++s) issued[s] = 0, issued_phase[s] = 0;
    bool alive = true;
    // QA: A copies of the first stages wait for the gate (B goes out first)
    bool gate_open = !QA;
    int n_def = 0, n_issued = 0;
    uint32_t def_stage[kStages];
    int def_kb[kStages], def_row[kStages];
    auto open_gate = [&]() -> bool {
      bool ok = true;
      if (lane == 0) {
        ok = wait_gate(p.gate, gridDim.x, 2 * gridDim.x, p.ctl, abort_flag);
        for (int i = 0; ok && i < n_def; ++i)
          tma_load_2d(smem_u32(smem + def_stage[i] * C_::kStageBytes), &tmap_a, def_kb[i] * (BK / 2),
                      def_row[i], smem_u32(&sm->full[def_stage[i]]));
      }
      gate_open = true;
      n_def = 0;
      return __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
    };
    for (int t = cid; t < total_tiles && alive; t += ncl) {
      const TileInfo ti = tile_at(t);
      if (!ti.ok) continue;
      const uint32_t bytes = kABytes + C_::kBLoad;
      const int b_row = (GROUPED ? ti.e * (int)p.N : 0) + ti.n0;
      for (int kb = kb_begin; kb < kb_end; ++kb) {
        if (!gate_open && n_issued >= kStages && !open_gate()) {
          alive = false;
          break;
        }
        if (!mbar_wait(smem_u32(&sm->empty[stage]), phase ^ 1, p.ctl, abort_flag)) {
          alive = false;
          break;
        }
        uint8_t* st = smem + stage * C_::kStageBytes;
        const uint32_t full = smem_u32(&sm->full[stage]);
        if (lane == 0) {
          mbar_arrive_expect_tx(full, bytes);
          // A rows: the tile's rows (grouped: rows of the routed copy of the codes)
          if (gate_open) {
            tma_load_2d(smem_u32(st), &tmap_a, kb * (BK / 2), ti.m_row0, full);
          } else {
            def_stage[n_def] = stage, def_kb[n_def] = kb, def_row[n_def] = ti.m_row0;
            ++n_def;
          }
          // B codes: the whole tile, or this CTA's 128-row half of the pair's tile
          tma_load_2d(smem_u32(st + kABytes), &tmap_b, kb * (BK / 2),
                      b_row + (P2 ? crank * (BNT / 2) : 0), full);
        }
        n_def = __shfl_sync(0xffffffffu, n_def, 0);
        ++n_issued;
        issued[stage] = 1;
        issued_phase[stage] = phase;
        if (++stage == kStages) stage = 0, phase ^= 1;
      }
    }
    if (!gate_open && alive) open_gate();  // fewer stages than the ring holds
    // drain: every copy this warp issued has landed before the CTA exits
    if (lane == 0) {
      KernelCtl drain = p.ctl;
      for (int s = 0; s < kStages; ++s)
        if (issued[s]) mbar_wait(smem_u32(&sm->full[s]), issued_phase[s], drain, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (in a pair only the even CTA issues; the odd CTA's warp 1 only holds TMEM)
    uint32_t stage = 0, phase = 0, tcount = 0;
    bool alive = true;
    if (lane == 0 && leader) {
      for (int t = cid; t < total_tiles && alive; t += ncl, ++tcount) {
        const TileInfo ti = tile_at(t);
        if (!ti.ok) { --tcount; continue; }
        if (!mbar_wait(smem_u32(&sm->acc_empty), (tcount & 1) ^ 1, p.ctl, abort_flag)) {
          alive = false;
          break;
        }
        tc_fence_after();
        for (int kb = kb_begin; kb < kb_end; ++kb) {
          // sf_full implies full in both CTAs: every scale-writer warp waits
          // for its own CTA's copies of the stage before it arrives
          if (!mbar_wait(smem_u32(&sm->sf_full[stage]), phase, p.ctl, abort_flag)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + stage * C_::kStageBytes);
          const uint32_t sf_t = tmem + kAccCols + stage * kSfColsPerStage;
#pragma unroll
          for (uint32_t k = 0; k < BK / 64; ++k) {
            const uint64_t ad = smem_desc(st + 32 * k, 16, 1024, 2);
            const uint64_t bd = smem_desc(st + kABytes + 32 * k, 16, 1024, 2);
            const uint32_t j = NV ? k : k >> 1;
            const uint32_t sf_id = NV ? 0u : (k & 1) * 2;
            const uint32_t idesc = fp4_idesc(BM * TM, BNT, !NV, sf_id, sf_id);
            const uint32_t acc = (kb != kb_begin || k != 0) ? 1u : 0u;
            if constexpr (P2)
              tc_mma_fp4_pair<NV ? 4 : 2>(tmem, ad, bd, idesc, sf_t + 4 * j, sf_t + 16 + 8 * j, acc);
            else
              tc_mma_fp4<NV ? 4 : 2>(tmem, ad, bd, idesc, sf_t + 4 * j, sf_t + 16 + 8 * j, acc);
          }
          // the stage is free in both CTAs once these MMAs are done
          if constexpr (P2) tc_commit_pair_mc(smem_u32(&sm->empty[stage]), 3);
          else tc_commit(smem_u32(&sm->empty[stage]));
          if (++stage == kStages) stage = 0, phase ^= 1;
        }
        if (!alive) break;
        if constexpr (P2) tc_commit_pair_mc(smem_u32(&sm->acc_full), 3);
        else tc_commit(smem_u32(&sm->acc_full));
      }
      // all MMAs this thread issued are complete before TMEM is released
      if constexpr (P2) tc_commit_pair_mc(smem_u32(&sm->mma_done), 1);
      else tc_commit(smem_u32(&sm->mma_done));
      KernelCtl drain = p.ctl;
      mbar_wait(smem_u32(&sm->mma_done), 0, drain, nullptr);
    }
    __syncwarp();
  } else if (warp >= kWriterWarp0 && warp < kWriterWarp0 + 4) {
    // ------------------------------------------------------------ scale writers
    // TMEM scale layout (the one tcgen05.cp .32x128b.warpx4 produces): chunk j
    // of A (512 bytes: 32 rows of 16) at columns 4j..4j+3, chunk j of B rows
    // h*128.. at columns 16 + 8j + 4h..; lane 32 q + l of every lane quarter q
    // holds the chunk's row l.  This warp writes its quarter's lanes.
    const int q = warp & 3;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t stage = 0, phase = 0;
    bool alive = true;
    for (int t = cid; t < total_tiles && alive; t += ncl) {
      const TileInfo ti = tile_at(t);
      if (!ti.ok) continue;
      for (int kb = kb_begin; kb < kb_end; ++kb) {
        if (!mbar_wait(smem_u32(&sm->full[stage]), phase, p.ctl, abort_flag)) {
          alive = false;
          break;
        }
        // the MMAs that last read this stage's scale columns completed before
        // the stage was refilled (empty -> producer -> full)
        tc_fence_after();
        const uint8_t* sfa_s = smem + stage * C_::kStageBytes + C_::kSfaOff;
        const uint8_t* sfb_s = smem + stage * C_::kStageBytes + C_::kSfbOff;
        const uint32_t sf_t = tmem + lane_base + kAccCols + stage * kSfColsPerStage;
#pragma unroll
        for (uint32_t j = 0; j < C_::kSfChunks; ++j) {
          const uint4 va = *reinterpret_cast<const uint4*>(sfa_s + 512 * j + 16 * lane);
          const uint4 vb0 = *reinterpret_cast<const uint4*>(sfb_s + 512 * j + 16 * lane);
          const uint4 vb1 = *reinterpret_cast<const uint4*>(sfb_s + C_::kSfaBytes + 512 * j + 16 * lane);
          tmem_st_32x32b_x4(sf_t + 4 * j, va);
          tmem_st_32x32b_x4(sf_t + 16 + 8 * j, vb0);
          tmem_st_32x32b_x4(sf_t + 16 + 8 * j + 4, vb1);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_leader(&sm->sf_full[stage]);
        if (++stage == kStages) stage = 0, phase ^= 1;
      }
    }
  } else if (warp == kWriterWarp0 + 4) {
    // ------------------------------------------------------------ scale producer
    // (the same walk over tiles and stages as the code producer)
    uint32_t stage = 0, phase = 0;
    int issued[kStages];
    uint32_t issued_phase[kStages];
    for (int s = 0; s < kStages; ++s) issued[s] = 0, issued_phase[s] = 0;
    bool alive = true;
    const int nsf4_a = (int)((p.K / (NV ? 16 : 32) + 3) / 4);
    const int nblk_b = (int)((p.N + 127) / 128);
    // QA: A scale copies of the first stages wait for the gate
    bool gate_open = !QA;
    int n_def = 0, n_issued = 0;
    uint32_t def_stage[kStages];
    const uint8_t* def_src[kStages];
    auto open_gate = [&]() -> bool {
      bool ok = true;
      if (lane == 0) {
        ok = wait_gate(p.gate, gridDim.x, 2 * gridDim.x, p.ctl, abort_flag);
        for (int i = 0; ok && i < n_def; ++i)
          bulk_load(smem_u32(smem + def_stage[i] * C_::kStageBytes + C_::kSfaOff), def_src[i],
                    C_::kSfaBytes, smem_u32(&sm->full[def_stage[i]]));
      }
      gate_open = true;
      n_def = 0;
      return __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
    };
    for (int t = cid; t < total_tiles && alive; t += ncl) {
      const TileInfo ti = tile_at(t);
      if (!ti.ok) continue;
      const bool a_sf_ok = ti.sf_block < (GROUPED ? (1 << 30) : p.num_m);  // a CTA past M loads no scales
      const uint8_t* sfa = p.a_sf + (int64_t)ti.sf_block * nsf4_a * 512;
      const uint8_t* sfb = p.b_sf + (int64_t)ti.e * p.b_sf_expert_bytes;
      const int nb0 = ti.n0 / 128;
      const bool b_hi = BNT > 128 && nb0 + 1 < nblk_b;  // the tile's second 128 B rows exist
      const uint32_t bytes = (a_sf_ok ? C_::kSfaBytes : 0u) + C_::kSfaBytes * (b_hi ? 2 : 1);
      for (int kb = kb_begin; kb < kb_end; ++kb) {
        if (!gate_open && n_issued >= kStages && !open_gate()) {
          alive = false;
          break;
        }
        if (!mbar_wait(smem_u32(&sm->empty[stage]), phase ^ 1, p.ctl, abort_flag)) {
          alive = false;
          break;
        }
        uint8_t* st = smem + stage * C_::kStageBytes;
        const uint32_t full = smem_u32(&sm->full[stage]);
        if (lane == 0) {
          mbar_arrive_expect_tx(full, bytes);
          const int64_t jsf = (int64_t)kb * C_::kSfChunks * 512;
          if (a_sf_ok) {
            if (gate_open) {
              bulk_load(smem_u32(st + C_::kSfaOff), sfa + jsf, C_::kSfaBytes, full);
            } else {
              def_stage[n_def] = stage, def_src[n_def] = sfa + jsf;
              ++n_def;
            }
          }
          const uint8_t* sfb0 = sfb + (int64_t)nb0 * nsf4_a * 512 + jsf;
          const uint32_t sfb_s = smem_u32(st + C_::kSfbOff);
          bulk_load(sfb_s, sfb0, C_::kSfaBytes, full);
          if (b_hi) bulk_load(sfb_s + C_::kSfaBytes, sfb0 + nsf4_a * 512, C_::kSfaBytes, full);
        }
        n_def = __shfl_sync(0xffffffffu, n_def, 0);
        ++n_issued;
        issued[stage] = 1;
        issued_phase[stage] = phase;
        if (++stage == kStages) stage = 0, phase ^= 1;
      }
    }
    if (!gate_open && alive) open_gate();  // fewer stages than the ring holds
    if (lane == 0) {
      KernelCtl drain = p.ctl;
      for (int s = 0; s < kStages; ++s)
        if (issued[s]) mbar_wait(smem_u32(&sm->full[s]), issued_phase[s], drain, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint32_t tcount = 0;
    for (int t = cid; t < total_tiles; t += ncl) {
      const TileInfo ti = tile_at(t);
      if (!ti.ok) continue;
      if (!mbar_wait(smem_u32(&sm->acc_full), tcount & 1, p.ctl, abort_flag)) break;
      tc_fence_after();
      if constexpr (KS > 1) {
        if (p.part_g) {
          // split-K through L2: this CTA's FP32 partial tile -> its slot of the
          // workspace, [BNT / 4][BM] float4 (a warp stores 512 contiguous bytes)
          const bool has_k = kb_end > kb_begin;
          float4* dst = p.part_g + (size_t)(cid * KS + krank) * (BNT / 4) * BM + (q * 32 + lane);
#pragma unroll 1
          for (int c0 = 0; c0 < BNT / 32; c0 += 4) {  // four 32-column loads per TMEM wait
            uint32_t r[4][32];
#pragma unroll
            for (int g = 0; g < 4; ++g)
              tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + (c0 + g) * 32, r[g]);
            tmem_ld_wait();
#pragma unroll
            for (int g = 0; g < 4; ++g)
#pragma unroll
              for (int v = 0; v < 8; ++v)
                dst[(size_t)((c0 + g) * 8 + v) * BM] =
                    has_k ? make_float4(__uint_as_float(r[g][4 * v]), __uint_as_float(r[g][4 * v + 1]),
                                        __uint_as_float(r[g][4 * v + 2]), __uint_as_float(r[g][4 * v + 3]))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
          }
          tc_fence_before();
          ++tcount;
          continue;
        }
        // split-K: this CTA's FP32 partial tile -> shared memory (the ring is idle:
        // every copy of this CTA's K slice was consumed before acc_full)
        float* part = reinterpret_cast<float*>(smem) + (q * 32 + lane) * kPartStride;
        const bool has_k = kb_end > kb_begin;
#pragma unroll 1
        for (int c0 = 0; c0 < BNT / 32; c0 += 4) {  // four 32-column loads per TMEM wait
          uint32_t r[4][32];
#pragma unroll
          for (int g = 0; g < 4; ++g)
            tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + (c0 + g) * 32, r[g]);
          tmem_ld_wait();
#pragma unroll
          for (int g = 0; g < 4; ++g)
#pragma unroll
            for (int v = 0; v < 8; ++v)
              reinterpret_cast<float4*>(part + (c0 + g) * 32)[v] =
                  has_k ? make_float4(__uint_as_float(r[g][4 * v]), __uint_as_float(r[g][4 * v + 1]),
                                      __uint_as_float(r[g][4 * v + 2]), __uint_as_float(r[g][4 * v + 3]))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        tc_fence_before();
        ++tcount;
        continue;
      }
      float alpha = 1.f;
      if constexpr (NV) alpha = __ldg(p.a_g) * __ldg(p.b_g + ti.e);
      const int row = ti.m_row0 + q * 32 + lane;
      const bool row_ok = row < ti.m_end;
      const bool vec_ok = (p.N % 8) == 0;
      auto store_chunk = [&](int c, const uint32_t (&r)[32]) {
        const int col0 = ti.n0 + c * 32;
        if (!row_ok || col0 >= p.N) return;
        const bool full_chunk = col0 + 32 <= p.N;
        if (p.c_dtype == Q4_BF16) {
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.C) + (int64_t)row * p.N + col0;
          if (full_chunk && vec_ok) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t w[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(
                    __uint_as_float(r[v * 8 + 2 * i]) * alpha,
                    __uint_as_float(r[v * 8 + 2 * i + 1]) * alpha);
                w[i] = *reinterpret_cast<const uint32_t*>(&h);
              }
              reinterpret_cast<uint4*>(out)[v] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (col0 + i < p.N) out[i] = __float2bfloat16_rn(__uint_as_float(r[i]) * alpha);
          }
        } else {
          float* out = reinterpret_cast<float*>(p.C) + (int64_t)row * p.N + col0;
          if (full_chunk && (p.N % 4) == 0) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              reinterpret_cast<float4*>(out)[v] =
                  make_float4(__uint_as_float(r[4 * v]) * alpha, __uint_as_float(r[4 * v + 1]) * alpha,
                              __uint_as_float(r[4 * v + 2]) * alpha, __uint_as_float(r[4 * v + 3]) * alpha);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (col0 + i < p.N) out[i] = __uint_as_float(r[i]) * alpha;
          }
        }
      };
      // Four 32-column TMEM loads per wait; the accumulator goes back to the
      // MMA as soon as its last columns are in registers, before they are
      // scaled and stored.
      const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < BNT / 32; c0 += 4) {
        uint32_t r[4][32];
#pragma unroll
        for (int g = 0; g < 4; ++g) tmem_ld_32x32b_x32(t_row + (c0 + g) * 32, r[g]);
        tmem_ld_wait();
        if (c0 + 4 >= BNT / 32) {  // every accumulator column is in registers
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_leader(&sm->acc_empty);
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) store_chunk(c0 + g, r[g]);
      }
      ++tcount;
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (P2) cluster_barrier_sync();  // the pair's MMAs are complete in both CTAs
  if (warp == 1) {
    tc_fence_after();
    if constexpr (P2) tmem_dealloc_pair(tmem, kTmemCols);
    else tmem_dealloc(tmem, kTmemCols);
  }
  if constexpr (KS > 1) {
   if (p.part_g) {
    // rank q reduces rows [q * 128 / KS, (q + 1) * 128 / KS) of the tile over
    // all ranks' partials in L2, in rank order, applies gA * gB and stores.
    // The cluster barrier (release / acquire at cluster scope) orders every
    // rank's partial stores before these loads; no CTA touches another's
    // shared memory, so none waits for the others afterwards.
    float alpha = 1.f;
    if constexpr (NV) alpha = __ldg(p.a_g) * __ldg(p.b_g);
    cluster_barrier_sync();
    const int t = cid;  // one tile per cluster
    if (t < total_tiles && !*abort_flag) {
      const TileInfo ti = tile_at(t);
      const int rows = (BM + KS - 1) / KS;
      const int r_lo = krank * rows, r_hi = min(BM, r_lo + rows);
      const int nr = r_hi - r_lo;
      const float4* src = p.part_g + (size_t)cid * KS * (BNT / 4) * BM;
      for (int e = threadIdx.x; e < nr * (BNT / 4); e += blockDim.x) {
        const int c4 = e / nr, r = r_lo + e % nr;  // consecutive threads: consecutive rows
        float4 sum = __ldcg(src + (size_t)c4 * BM + r);
#pragma unroll
        for (int qq = 1; qq < KS; ++qq) {
          const float4 v = __ldcg(src + (size_t)(qq * (BNT / 4) + c4) * BM + r);
          sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
        }
        const int row = ti.m_row0 + r, col = ti.n0 + 4 * c4;
        if (row >= ti.m_end || col >= p.N) continue;
        const float o[4] = {sum.x * alpha, sum.y * alpha, sum.z * alpha, sum.w * alpha};
        if (p.c_dtype == Q4_BF16) {
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.C) + (int64_t)row * p.N + col;
          if (col + 4 <= p.N && (p.N % 4) == 0) {  // 8-byte aligned: one store
            const __nv_bfloat162 lo = __floats2bfloat162_rn(o[0], o[1]), hi = __floats2bfloat162_rn(o[2], o[3]);
            uint2 w;
            w.x = *reinterpret_cast<const uint32_t*>(&lo);
            w.y = *reinterpret_cast<const uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(out) = w;
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (col + i < p.N) out[i] = __float2bfloat16_rn(o[i]);
          }
        } else {
          float* out = reinterpret_cast<float*>(p.C) + (int64_t)row * p.N + col;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (col + i < p.N) out[i] = o[i];
        }
      }
    }
    return;
   }
    // rank q reduces rows [q * 128 / KS, (q + 1) * 128 / KS) of the tile over all
    // ranks' partials, in rank order, then applies gA * gB and stores
    float alpha = 1.f;
    if constexpr (NV) alpha = __ldg(p.a_g) * __ldg(p.b_g);  // loaded before the barrier
    cluster_barrier_sync();
    const int t = cid;  // one tile per cluster
    if (t < total_tiles && !*abort_flag) {
      const TileInfo ti = tile_at(t);
      const int rows = (BM + KS - 1) / KS;
      const int r_lo = krank * rows, r_hi = min(BM, r_lo + rows);
      const uint32_t base = smem_u32(smem);
      const int items = (r_hi - r_lo) * (BNT / 4);
      // kBatch items per thread per round: all their remote loads are in flight
      // together, so a round costs one distributed-shared-memory round trip
      constexpr int kBatch = 4;
      for (int e0 = threadIdx.x; e0 < items; e0 += kBatch * blockDim.x) {
        float4 v[kBatch][KS];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int e = e0 + b * blockDim.x;
          const int r = r_lo + (e < items ? e : 0) / (BNT / 4), c4 = (e < items ? e : 0) % (BNT / 4);
          const uint32_t off = (uint32_t)(r * kPartStride + 4 * c4) * 4u;
#pragma unroll
          for (int qq = 0; qq < KS; ++qq)  // this CTA's own partial by a plain shared load
            v[b][qq] = qq == krank ? *reinterpret_cast<const float4*>(smem + off)
                                   : ld_dsmem_v4(base + off, (uint32_t)qq);
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int e = e0 + b * blockDim.x;
          if (e >= items) break;
          const int r = r_lo + e / (BNT / 4), c4 = e % (BNT / 4);
          float4 sum = v[b][0];
#pragma unroll
          for (int qq = 1; qq < KS; ++qq) {
            sum.x += v[b][qq].x; sum.y += v[b][qq].y; sum.z += v[b][qq].z; sum.w += v[b][qq].w;
          }
          const int row = ti.m_row0 + r, col = ti.n0 + 4 * c4;
          if (row >= ti.m_end || col >= p.N) continue;
          const float o[4] = {sum.x * alpha, sum.y * alpha, sum.z * alpha, sum.w * alpha};
          if (p.c_dtype == Q4_BF16) {
            __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.C) + (int64_t)row * p.N + col;
            if (col + 4 <= p.N && (p.N % 4) == 0) {  // 8-byte aligned: one store
              const __nv_bfloat162 lo = __floats2bfloat162_rn(o[0], o[1]), hi = __floats2bfloat162_rn(o[2], o[3]);
              uint2 w;
              w.x = *reinterpret_cast<const uint32_t*>(&lo);
              w.y = *reinterpret_cast<const uint32_t*>(&hi);
              *reinterpret_cast<uint2*>(out) = w;
            } else {
#pragma unroll
              for (int i = 0; i < 4; ++i)
                if (col + i < p.N) out[i] = __float2bfloat16_rn(o[i]);
            }
          } else {
            float* out = reinterpret_cast<float*>(p.C) + (int64_t)row * p.N + col;
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (col + i < p.N) out[i] = o[i];
          }
        }
      }
    }
  }
  // no CTA leaves while its peer may still commit to it, arrive on its
  // barriers or read its shared memory
  if constexpr (CL > 1) cluster_barrier_sync();
}

// ------------------------------------------------------------------ grouped prep
// sched[e] = first tile-row of expert e (prefix of ceil(M_e / 128)).
__global__ void grouped_sched_kernel(const int32_t* __restrict__ offsets, int E,
                                     int32_t* __restrict__ sched) {
  pdl_wait();
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    int acc = 0;
    sched[0] = 0;
    for (int e = 0; e < E; ++e) {
      const int m = __ldg(offsets + e + 1) - __ldg(offsets + e);
      acc += (max(m, 0) + BM - 1) / BM;
      sched[e + 1] = acc;
    }
  }
}

// Routed A scales in the tensor-core layout: tile-row tr, local row i holds
// the scales of token row_token[offsets[e] + (tr - sched[e]) * 128 + i]
// (zero past the expert's last row).  One block of 128 threads per tile-row,
// thread i = local row i.  Each pass moves 8 scale tiles (32 bytes of every
// row's scales): two 16-byte loads per thread, a transpose in shared memory,
// then 4096 contiguous bytes out as 16-byte stores.  nsf is a multiple of 16
// (K % 256 == 0), so every token's scale row is 16-byte aligned.
__global__ void __launch_bounds__(128)
    grouped_sf_kernel(const int32_t* __restrict__ offsets, const int32_t* __restrict__ row_token,
                      const int32_t* __restrict__ sched, int E,
                      const uint8_t* __restrict__ tok_sf, int64_t nsf,
                      uint8_t* __restrict__ out) {
  pdl_wait();
  __shared__ uint4 tiles[8 * 32];  // 8 tiles of 512 bytes
  uint32_t* tw = reinterpret_cast<uint32_t*>(tiles);
  const int tr = blockIdx.x;
  if (tr >= __ldg(sched + E)) return;
  int e = 0;
  while (e + 1 < E && __ldg(sched + e + 1) <= tr) ++e;
  const int i = threadIdx.x;
  const int r = __ldg(offsets + e) + (tr - __ldg(sched + e)) * BM + i;
  const bool ok = r < __ldg(offsets + e + 1);
  const uint4* src =
      ok ? reinterpret_cast<const uint4*>(tok_sf + (int64_t)__ldg(row_token + r) * nsf) : nullptr;
  const int64_t nsf4 = nsf / 4;  // 4-scale columns: tiles per tile-row (a multiple of 4)
  uint4* dst = reinterpret_cast<uint4*>(out + (int64_t)tr * nsf4 * 512);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  // word of row i inside a tile: byte (i % 32) * 16 + (i / 32) * 4
  const int wi = (i & 31) * 4 + (i >> 5);
  for (int64_t J0 = 0; J0 < nsf4; J0 += 8) {
    const int nj = nsf4 - J0 < 8 ? 4 : 8;  // nsf4 is a multiple of 4
    const uint4 v0 = ok ? __ldg(src + J0 / 4) : zero;
    const uint4 v1 = ok && nj > 4 ? __ldg(src + J0 / 4 + 1) : zero;
    tw[0 * 128 + wi] = v0.x;
    tw[1 * 128 + wi] = v0.y;
    tw[2 * 128 + wi] = v0.z;
    tw[3 * 128 + wi] = v0.w;
    tw[4 * 128 + wi] = v1.x;
    tw[5 * 128 + wi] = v1.y;
    tw[6 * 128 + wi] = v1.z;
    tw[7 * 128 + wi] = v1.w;
    __syncthreads();
    for (int v = i; v < nj * 32; v += 128) dst[J0 * 32 + v] = tiles[v];
    __syncthreads();
  }
}
}  // namespace

namespace {

// Routed copy of the token codes: out[r] = codes[row_token[r]], r < R, so that
// each expert's routed rows are consecutive and reach the GEMM by TMA.
// 16-byte vectors, grid-stride; row_bytes is a multiple of 16.
__global__ void __launch_bounds__(256)
    gather_rows_kernel(const uint8_t* __restrict__ codes, const int32_t* __restrict__ row_token,
                       int64_t R, int64_t row_bytes, uint8_t* __restrict__ out) {
  pdl_wait();
  const int64_t vpr = row_bytes / 16, total = R * vpr;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total;
       v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = v / vpr, c = v - r * vpr;
    const int64_t tok = __ldg(row_token + r);
    reinterpret_cast<uint4*>(out)[v] = __ldg(reinterpret_cast<const uint4*>(codes + tok * row_bytes) + c);
  }
}

template <bool NV, bool GROUPED, int KS = 1, bool P2 = false, int BNT = BN, bool QA = false>
q4_status set_smem_attr() {
  static int done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return Q4_ERR_CUDA;
  if (!done[dev]) {
    Q4_CUDA_TRY(cudaFuncSetAttribute(fp4_gemm_kernel<NV, GROUPED, KS, P2, BNT, QA>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)Cfg<NV, P2, BNT>::kSmemBytes));
    done[dev] = 1;
  }
  return Q4_OK;
}

// Persistent dense launch: single CTAs, or CTA pairs (P2) on 256x256 tiles.
template <bool NV, bool P2, bool QA = false>
q4_status launch_dense(const CUtensorMap& ta, const CUtensorMap& tb, const Params& p,
                       cudaStream_t stream) {
  q4_status st;
  if ((st = set_smem_attr<NV, false, 1, P2, BN, QA>()) != Q4_OK) return st;
  constexpr int CL = P2 ? 2 : 1;
  const int ctiles = ((p.num_m + CL - 1) / CL) * p.num_n;  // cluster tiles
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(block_threads<false>(), 1, 1);
  cfg.dynamicSmemBytes = Cfg<NV, P2>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the kernel waits (griddepcontrol.wait)
  // before touching memory the previous kernel may have written
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // persistent clusters: exactly as many as can be resident at once, so no
  // cluster waits for a second wave with its whole share of tiles
  static int max_active[64][2] = {{0}};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return Q4_ERR_CUDA;
  if (!max_active[dev][P2]) {
    int n = 0;
    cfg.gridDim = dim3((unsigned)(num_sms() / CL * CL), 1, 1);
    if (cudaOccupancyMaxActiveClusters(&n, fp4_gemm_kernel<NV, false, 1, P2, BN, QA>, &cfg) != cudaSuccess || n <= 0)
      n = num_sms() / CL;
    max_active[dev][P2] = std::min(n, num_sms() / CL);
  }
  const int clusters = std::max(1, std::min(ctiles, max_active[dev][P2]));
  cfg.gridDim = dim3((unsigned)(clusters * CL), 1, 1);
  Q4_CUDA_TRY(cudaLaunchKernelEx(&cfg, fp4_gemm_kernel<NV, false, 1, P2, BN, QA>, ta, tb, p));
  return Q4_OK;
}

// Split-K for problems with few output tiles: KS CTAs (one cluster) per tile,
// launched as exactly tiles x KS CTAs (one tile per cluster).
template <bool NV, int KS, int BNT, bool QA = false>
q4_status launch_splitk(const CUtensorMap& ta, const CUtensorMap& tb, const Params& p,
                        cudaStream_t stream) {
  using C_ = Cfg<NV, false, BNT>;
  static_assert(KS * 0 + (BM * C_::kPartStride * 4) <= C_::kStages * C_::kStageBytes, "partial tile fits");
  q4_status st;
  if ((st = set_smem_attr<NV, false, KS, false, BNT, QA>()) != Q4_OK) return st;
  const int tiles = p.num_m * p.num_n;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * KS), 1, 1);
  cfg.blockDim = dim3(block_threads<false>(), 1, 1);
  cfg.dynamicSmemBytes = C_::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = KS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the kernel waits (griddepcontrol.wait)
  // before touching memory the previous kernel may have written
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  Q4_CUDA_TRY(cudaLaunchKernelEx(&cfg, fp4_gemm_kernel<NV, false, KS, false, BNT, QA>, ta, tb, p));
  return Q4_OK;
}

// Whether `clusters` clusters of KS CTAs of this split-K instantiation can all
// be resident at once (the QA prologue's gate needs every CTA running).
template <bool NV, int KS, int BNT>
bool splitk_resident(int clusters) {
  using C_ = Cfg<NV, false, BNT>;
  if (set_smem_attr<NV, false, KS, false, BNT, true>() != Q4_OK) return false;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(clusters * KS), 1, 1);
  cfg.blockDim = dim3(block_threads<false>(), 1, 1);
  cfg.dynamicSmemBytes = C_::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = KS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  return cudaOccupancyMaxActiveClusters(&n, fp4_gemm_kernel<false, false, KS, false, BNT, true>, &cfg) ==
             cudaSuccess &&
         n >= clusters;
}

template <bool NV, int BNT, bool QA = false>
q4_status dispatch_splitk(int ks, const CUtensorMap& ta, const CUtensorMap& tb, const Params& p,
                          cudaStream_t stream) {
  switch (ks) {  // 2 <= ks <= 4
    case 2: return launch_splitk<NV, 2, BNT, QA>(ta, tb, p, stream);
    case 3: return launch_splitk<NV, 3, BNT, QA>(ta, tb, p, stream);
    default: return launch_splitk<NV, 4, BNT, QA>(ta, tb, p, stream);
  }
}


}  // namespace

// Workspace bytes for the split-K partial sums of an M x N x K FP4 GEMM: the
// most the launch below can take (clusters of up to 4 CTAs), 0 when the shape
// does not split K.  nsms: the SM count the launch will see.
size_t fp4_splitk_partial_bytes(int64_t M, int64_t N, int64_t K, int nsms) {
  if (M <= 0 || N <= 0 || K / BK < 2) return 0;
  const int64_t num_m = ceil_div(M, BM);
  const int64_t t128 = num_m * ceil_div(N, 128), t256 = num_m * ceil_div(N, (int64_t)BN);
  if (t128 * 2 <= nsms) return (size_t)t128 * 4 * BM * 128 * sizeof(float);
  if (t256 * 2 <= nsms) return (size_t)t256 * 4 * BM * BN * sizeof(float);
  return 0;
}

q4_status launch_fp4_gemm(const Fp4GemmArgs& a, cudaStream_t stream) {
  if (a.M == 0 || a.N == 0) return Q4_OK;
  CUtensorMap ta, tb;
  q4_status st;
  if ((st = make_tmap_2d_u8(&ta, a.a_codes, a.K / 2, a.M, a.K / 2, BK / 2, BM, true)) != Q4_OK) return st;
  if ((st = make_tmap_2d_u8(&tb, a.b_codes, a.K / 2, a.N, a.K / 2, BK / 2, BN, true)) != Q4_OK) return st;
  Params p = {};
  p.M = a.M; p.N = a.N; p.K = a.K;
  p.a_sf = a.a_scales; p.b_sf = a.b_scales; p.b_sf_expert_bytes = 0;
  p.a_g = a.a_g; p.b_g = a.b_g;
  p.C = a.C; p.c_dtype = a.c_dtype;
  p.num_m = (int)ceil_div(a.M, BM); p.num_n = (int)ceil_div(a.N, BN); p.bn = BN;
  p.ctl.status = device_status_ptr();
  p.ctl.wait_ns = wait_budget_ns();
  bool qa = a.a_raw != nullptr;  // MXFP4 activations quantized in the prologue
  if (qa) {
    if (a.nvfp4) return Q4_ERR_INVALID_ARG;
    // split-K runs the prologue only when every cluster is resident at once;
    // otherwise the activations are quantized by a separate pass first
    const int nkb = (int)(a.K / BK);
    const int t128 = p.num_m * (int)ceil_div(a.N, 128), t256 = p.num_m * p.num_n;
    int ks = 0, tiles = 0;
    bool n128 = false;
    if (t128 * 2 <= num_sms() && nkb >= 2) ks = std::min(4, std::min(num_sms() / t128, nkb)), tiles = t128, n128 = true;
    else if (t256 * 2 <= num_sms() && nkb >= 2) ks = std::min(4, std::min(num_sms() / t256, nkb)), tiles = t256;
    if (ks >= 2) {
      bool fits;
      if (n128) fits = ks == 2 ? splitk_resident<false, 2, 128>(tiles) : ks == 3 ? splitk_resident<false, 3, 128>(tiles)
                                                                               : splitk_resident<false, 4, 128>(tiles);
      else fits = ks == 2 ? splitk_resident<false, 2, BN>(tiles) : ks == 3 ? splitk_resident<false, 3, BN>(tiles)
                                                                         : splitk_resident<false, 4, BN>(tiles);
      if (!fits) {
        if ((st = launch_quant_mxfp4(a.a_raw, a.a_dtype, a.M, a.K, const_cast<uint8_t*>(a.a_codes),
                                     const_cast<uint8_t*>(a.a_scales), Q4_SCALES_MMA, stream)) != Q4_OK)
          return st;
        qa = false;
      }
    }
  }
  if (qa) {
    p.a_raw = a.a_raw;
    p.a_dtype = a.a_dtype;
    p.a_codes_w = const_cast<uint8_t*>(a.a_codes);
    p.a_sf_w = const_cast<uint8_t*>(a.a_scales);
    p.gate = a.gate;
  }
  // few output tiles: split K over a cluster so that the grid fills the GPU,
  // on 128-wide N tiles when there are few enough of them (twice the tiles,
  // half the bytes and half the partial tile per CTA).  At most 4 CTAs per
  // cluster: measured on GB300 (256 x 2048 x 7168, 128 x 4096 x 8192) 4 is
  // fastest and 8 is slower than no split, since clusters of 8
  // one-CTA-per-SM blocks are not all resident at once.
  const int nkb = (int)(a.K / BK);
  const int tiles128 = p.num_m * (int)ceil_div(a.N, 128), tiles = p.num_m * p.num_n;
  // split-K partials meet in L2 when the caller's workspace holds them
  auto part_ws = [&](int t, int ks, int bnt) -> float4* {
    const size_t need = (size_t)t * ks * BM * bnt * sizeof(float);
    return a.part_ws && a.part_ws_bytes >= need ? static_cast<float4*>(a.part_ws) : nullptr;
  };
  if (tiles128 * 2 <= num_sms() && nkb >= 2) {
    const int ks = std::min(4, std::min(num_sms() / tiles128, nkb));
    CUtensorMap tb128;
    if ((st = make_tmap_2d_u8(&tb128, a.b_codes, a.K / 2, a.N, a.K / 2, BK / 2, 128, true)) != Q4_OK) return st;
    Params p128 = p;
    p128.num_n = (int)ceil_div(a.N, 128);
    p128.bn = 128;
    p128.part_g = part_ws(tiles128, ks, 128);
    if (qa) return dispatch_splitk<false, 128, true>(ks, ta, tb128, p128, stream);
    return a.nvfp4 ? dispatch_splitk<true, 128>(ks, ta, tb128, p128, stream)
                   : dispatch_splitk<false, 128>(ks, ta, tb128, p128, stream);
  }
  if (tiles * 2 <= num_sms() && nkb >= 2) {
    const int ks = std::min(4, std::min(num_sms() / tiles, nkb));
    if (ks >= 2) {
      p.part_g = part_ws(tiles, ks, BN);
      if (qa) return dispatch_splitk<false, BN, true>(ks, ta, tb, p, stream);
      return a.nvfp4 ? dispatch_splitk<true, BN>(ks, ta, tb, p, stream)
                     : dispatch_splitk<false, BN>(ks, ta, tb, p, stream);
    }
  }
  // CTA pairs (2-SM MMA on 256x256 tiles) whenever M spans two tiles: each SM
  // then receives half of each B tile
  if (p.num_m >= 2) {
    CUtensorMap tb2;  // 128-row boxes: each CTA loads its half of the B tile
    if ((st = make_tmap_2d_u8(&tb2, a.b_codes, a.K / 2, a.N, a.K / 2, BK / 2, BN / 2, true)) != Q4_OK) return st;
    if (qa) return launch_dense<false, true, true>(ta, tb2, p, stream);
    return a.nvfp4 ? launch_dense<true, true>(ta, tb2, p, stream) : launch_dense<false, true>(ta, tb2, p, stream);
  }
  if (qa) return launch_dense<false, false, true>(ta, tb, p, stream);
  return a.nvfp4 ? launch_dense<true, false>(ta, tb, p, stream) : launch_dense<false, false>(ta, tb, p, stream);
}

q4_status launch_grouped_prep(const int32_t* offsets, const int32_t* row_token, int E,
                              const uint8_t* tok_scales_rowmajor, int64_t nsf, int32_t* sched,
                              uint8_t* a_sf_routed, int64_t sf_rows_cap, cudaStream_t stream) {
  q4_status st = launch_pdl(grouped_sched_kernel, 1, 32, 0, stream, offsets, E, sched);
  if (st != Q4_OK) return st;
  const int64_t cap_blocks = sf_rows_cap / BM;
  if (cap_blocks > 0)
    st = launch_pdl(grouped_sf_kernel, (unsigned)cap_blocks, 128, 0, stream, offsets, row_token, sched,
                    E, tok_scales_rowmajor, nsf, a_sf_routed);
  return st;
}

q4_status launch_gather_rows(const uint8_t* codes, const int32_t* row_token, int64_t R,
                             int64_t row_bytes, uint8_t* out, cudaStream_t stream) {
  if (R == 0) return Q4_OK;
  const int64_t total = R * (row_bytes / 16);
  const unsigned grid = (unsigned)std::min<int64_t>(ceil_div(total, 256), (int64_t)num_sms() * 8);
  return launch_pdl(gather_rows_kernel, grid, 256, 0, stream, codes, row_token, R, row_bytes, out);
}

q4_status launch_grouped_gemm(const GroupedArgs& a, cudaStream_t stream) {
  if (a.R == 0 || a.N == 0 || a.E == 0) return Q4_OK;
  if (a.E > kMaxExperts) return Q4_ERR_UNSUPPORTED_SHAPE;
  CUtensorMap tb;
  q4_status st;
  // B: the E stacked expert weights as one tensor; A: the routed copy of the
  // token codes, so a tile's rows are consecutive
  CUtensorMap ta;
  if ((st = make_tmap_2d_u8(&tb, a.w_codes, a.K / 2, (uint64_t)a.E * a.N, a.K / 2, BK / 2, BN, true)) != Q4_OK) return st;
  if ((st = make_tmap_2d_u8(&ta, a.a_routed, a.K / 2, (uint64_t)a.R, a.K / 2, BK / 2, BM, true)) != Q4_OK) return st;
  Params p = {};
  p.M = a.R; p.N = a.N; p.K = a.K;
  p.a_sf = a.a_sf_rows; p.b_sf = a.w_scales;
  p.b_sf_expert_bytes = (int64_t)mma_scales_bytes(a.N, a.K / 16);
  p.a_g = a.a_g; p.b_g = a.w_g;
  p.C = a.C; p.c_dtype = Q4_BF16;
  p.num_m = 0; p.num_n = (int)ceil_div(a.N, BN); p.bn = BN;
  p.offsets = a.offsets; p.sched = a.sched; p.E = a.E;
  p.ctl.status = device_status_ptr();
  p.ctl.wait_ns = wait_budget_ns();
  if ((st = set_smem_attr<true, true>()) != Q4_OK) return st;
  return launch_pdl(fp4_gemm_kernel<true, true>, (unsigned)num_sms(), block_threads<true>(),
                    Cfg<true>::kSmemBytes, stream, ta, tb, p);
}

}  // namespace q4
