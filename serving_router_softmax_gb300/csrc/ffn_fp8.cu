// moe_verify_ffn, tensor-core path for FP8 E4M3 weights with fp32 block scales
// (one scale per 128 x 128 block of each expert matrix).
//
// Same method as the bf16 path (the union's experts are each streamed from HBM
// once; EcoSpec write-up, sections 1-2), with the 8-bit operands fed straight
// to tcgen05.mma kind::f8f6f4:
//   * A = E4M3 weights exactly as stored: 128 rows x 128 reduction bytes per
//     k-block, TMA-loaded with the 128-byte swizzle.
//   * B = activations as two E4M3 matrices per row: with a per-row scale s,
//     a power of two that puts max |x| / s in [128, 256) (so the scaling is
//     exact), hi = e4m3(x / s) and lo = e4m3((x / s - hi) * 16), so that
//     x ~= s * (hi + lo / 16) with relative error near 2^-8.  hi and lo rows
//     are stacked, so one MMA of N = 2 * np produces both partial products.
//   * The weight block scale changes every 128 reduction elements, so every
//     k-block is multiplied into its own TMEM buffer (up to 16 in rotation, as
//     many as fit in the 512 columns) and the
//     epilogue warps promote it: acc += w_scale * s * (d_hi + d_lo / 16), in
//     fp32 registers.  In the down projection the buffers go in pairs: one
//     commit and one barrier round trip per two k-blocks (there the
//     per-k-block synchronisation, not the tensor pipe, is the tighter
//     resource at these small N; gate/up, with half as many buffers, keeps
//     one k-block per barrier).
//   * gate/up writes h = silu(gate) * up quantized the same way, with one
//     scale per (token, 128-row block of I), which is exactly one k-block of
//     the down projection.
// Stream-K partitioning over the layer's k-blocks and the last-arriver fixup
// of split tiles follow the bf16 kernel; the weighted combine is its own
// kernel afterwards.
#include <cuda_fp8.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "l2_prefetch.cuh"
#include "ffn_internal.cuh"
#include "tc_ptx.cuh"
#include "stream_k.cuh"
#include "fp8_quant.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;           // weight rows per tile (MMA M)
constexpr int kBK = 128;           // reduction elements (bytes) per k-block
constexpr int kABytes = kBM * kBK;  // 16 KB
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kNBMax = 16;         // TMEM promotion buffers (at most)
constexpr int kMaxNM = 32;         // padded token columns handled by this path
using fp8q::kLoScale;
using fp8q::pow2_scale;
using fp8q::split_e4m3;
constexpr uint64_t kWaitBudgetNs = 2000000000ull;
constexpr uint64_t kReadyBudgetNs = 100000ull;     // 100 us for the union handshake
constexpr int kBarRegion = 512;    // mbarriers + flags of the CTA
static_assert((2 * 12 + 2 * kNBMax + 1) * 8 + 5 * 4 <= kBarRegion, "barrier region too small");

struct Fp8Params {
  int T, k, E, cap;
  int M, K;             // rows of each expert matrix, reduction length
  int NM;               // padded token columns (16 or 32): the token-dense gate/up operand
  int Rh;               // rows of the quantized intermediate: expert u's token rows from u * NM
  int tiled, KS, stages, pdl;
  int NB;               // TMEM promotion buffers in rotation
  uint32_t tmem_cols;
  const int32_t* n_unique;
  const int32_t* unique;
  const int32_t* offsets;
  const int32_t* perm_token;
  const float* wscale;  // block scales of this matrix: [E][scale_rows][K/128]
  int scale_rows;       // gate/up: 2I/128 (gate blocks, then up blocks); down: H/128
  const float* bscale;  // gate/up: [NM] per token row; down: [K/128][hs_stride]
  uint8_t* hq_hi;       // gate/up output [Rh][M]
  uint8_t* hq_lo;
  float* hscale;        // gate/up output [M/128][hs_stride]
  int hs_stride;        // rows of hscale per k-block (Rh)
  float* o;             // down output [T*k][M]
  float* partials;      // [grid][2][2*NM][128]
  int32_t* tile_cnt;
  int32_t* dev_err;
  const int32_t* slot_of;  // expert -> weight slot (NULL: identity); block scales stay per expert id
  int n_slots;
  // Union-ready handshake with the layer-head kernel that gate/up follows
  // directly (as in the bf16 kernel); NULL when a prep kernel sits between.
  int32_t* ready_flag;
  int32_t ready_value;
  int32_t* ready_clear;
  // down only: the next layer's predicted experts, which each CTA asks L2
  // to fetch (its round-robin share) once it has issued its last weight load.
  NextLayerPrefetch pf;
};

struct Tile {
  int u, m, e, ws, ne, np, prow, off;  // ws: the expert's slot in the weight buffers
  bool ok, prow_ok;
};

__device__ __forceinline__ Tile tile_info(const Fp8Params& p, int U, int t, bool with_prow) {
  Tile ti;
  ti.m = t / U;
  ti.u = t - ti.m * U;
  ti.e = p.unique[ti.u];
  ti.off = p.offsets[ti.u];
  ti.ne = p.offsets[ti.u + 1] - ti.off;
  ti.np = (ti.ne + 15) & ~15;
  ti.ok = ti.e >= 0 && ti.e < p.E && ti.ne >= 1 && ti.ne <= p.T && ti.np <= p.NM && ti.off >= 0 &&
          ti.off + ti.ne <= p.T * p.k;
  ti.ws = ti.ok ? weight_slot(p.slot_of, p.n_slots, ti.e) : -1;
  ti.ok = ti.ok && ti.ws >= 0;
  ti.prow = ti.u * p.NM;
  ti.prow_ok = ti.prow + p.NM <= p.Rh;
  (void)with_prow;
  return ti;
}

// silu(a) * b with the fast exponential and division (relative error near
// 1e-6, far below the 2^-8 of the E4M3 split that h goes through next); the
// tile end that calls it runs once per tile and is short for that reason.
__device__ __forceinline__ float silu_mul(float a, float b) { return __fdividef(a, 1.f + __expf(-a)) * b; }

// Instruction descriptor, kind::f8f6f4: D f32 (bits 4-5 = 1), A and B E4M3
// (format 0 in bits 7-9 and 10-12), both K-major, N >> 3 (17-22), M >> 4 (24-28).
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_e4m3(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <bool kGateUp>
__global__ void __launch_bounds__(kThreads, 1)
    ffn_fp8_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                   const __grid_constant__ CUtensorMap tmBhi, const __grid_constant__ CUtensorMap tmBlo,
                   const Fp8Params p) {
  constexpr int kGroup = kGateUp ? 1 : 2;  // k-blocks per TMEM barrier
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int aBytes = kGateUp ? 2 * kABytes : p.KS * kABytes;
  const int bStride = 2 * p.NM * 128;  // hi + lo rows of one k-block
  const int stageBytes = aBytes + p.KS * bStride;
  const int S = p.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + (size_t)S * stageBytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + kNBMax;
  uint64_t* drain = tempty + kNBMax;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* bcast = abort_flag + 1;
  volatile int* issued = bcast + 1;
  volatile int* consumed = issued + 1;
  // Barrier/flag block (at most 2*12 + 9 mbarriers + 5 words) then the combine's staging.
  float* s_red = reinterpret_cast<float*>(base + (size_t)S * stageBytes + kBarRegion);  // [4 warps][kMaxNM] column maxima
  float* s_sc = s_red + 4 * kMaxNM;  // [kMaxNM] 1 / scale of each column of h

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < p.NB / kGroup; ++b) {  // one group of TMEM buffers per barrier
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], kEpiThreads);
    }
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    *issued = 0;
    *consumed = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&tmA0);
    tc::tma_prefetch_desc(&tmA1);
    tc::tma_prefetch_desc(&tmBhi);
    tc::tma_prefetch_desc(&tmBlo);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_holder, p.tmem_cols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int MT = (p.M + kBM - 1) / kBM;
  const int KB = p.K / kBK;
  const int KU = (KB + p.KS - 1) / p.KS;
  const int c = blockIdx.x;
  int U = 0, G = 0;
  long long total = 0, s0 = 0, s1 = 0;
  // Splits the layer's pipeline units over at most `total` CTAs (see the
  // bf16 kernel); each role calls it once the union is visible to it.
  auto partition = [&](int u) {
    U = u;
    const bool valid = U >= 1 && U <= p.cap;
    total = valid ? (long long)U * MT * KU : 0;
    G = static_cast<int>(total < gridDim.x ? total : gridDim.x);
    s0 = c < G ? total * c / G : total;
    s1 = c < G ? total * (c + 1) / G : total;
  };
  auto load_partition = [&]() { partition(*p.n_unique); };
  if (!p.ready_flag) load_partition();  // complete before this grid started
  const uint32_t buf_cols = (kGateUp ? 4 : 2) * p.NM;  // per TMEM buffer: [gate hi|lo][up hi|lo]

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (tc::elect_one()) {
      const uint64_t polA = tc::policy_evict_first();
      const uint64_t polB = tc::policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int n_issued = 0;
      constexpr int kMaxPend = 16;
      int pend_t[kMaxPend], pend_kb[kMaxPend], pend_nq[kMaxPend], pend_st[kMaxPend];
      int npend = 0;
      bool dep_done = !p.pdl;
      if (dep_done) tc::griddep_launch_dependents();
      if (p.ready_flag) {
        // The union comes from the head kernel this grid follows directly:
        // read it early once the head has published it (acquire), else
        // after the dependency wait (see the bf16 kernel).
        int32_t word = 0;
        if (!dep_done && tc::wait_flag_acquire(p.ready_flag, p.ready_value, kReadyBudgetNs, &word)) {
          partition(static_cast<int>(static_cast<uint32_t>(word) >> 16));
        } else {
          if (!dep_done) {
            tc::griddep_wait();
            tc::griddep_launch_dependents();
            dep_done = true;
          }
          load_partition();
        }
      }
      auto issue_b = [&](int t, int kb, int nq, int st) {
        uint8_t* sB = base + (size_t)st * stageBytes + aBytes;
        if (kGateUp) {
          // token-dense: all NM token rows in one box each (rows past T read as zeros)
          tc::tma_load_2d(sB, &tmBhi, kb * kBK, 0, &full[st], polB);
          tc::tma_load_2d(sB + p.NM * 128, &tmBlo, kb * kBK, 0, &full[st], polB);
          return;
        }
        const Tile ti = tile_info(p, U, t, true);
        const int prow = ti.prow_ok ? ti.prow : 0;
        for (int q = 0; q < nq; ++q)
          for (int j = 0; j < ti.np / 16; ++j) {
            tc::tma_load_2d(sB + q * bStride + j * 2048, &tmBhi, (kb + q) * kBK, prow + 16 * j, &full[st], polB);
            tc::tma_load_2d(sB + q * bStride + ti.np * 128 + j * 2048, &tmBlo, (kb + q) * kBK, prow + 16 * j,
                            &full[st], polB);
          }
      };
      auto resolve = [&]() {
        tc::griddep_wait();
        tc::griddep_launch_dependents();
        for (int i = 0; i < npend; ++i) issue_b(pend_t[i], pend_kb[i], pend_nq[i], pend_st[i]);
        npend = 0;
        dep_done = true;
      };
      Segments sg;
      sg.init(s0, s1, KU, false);
      for (int si = 0; si < sg.n && !*abort_flag; ++si) {
        int t, u0, u1;
        sg.get(si, t, u0, u1);
        const Tile ti = tile_info(p, U, t, false);
        if (!ti.ok) continue;
        for (int uu = u0; uu < u1; ++uu) {
          if (!dep_done && npend == S) resolve();
          if (!tc::mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, kWaitBudgetNs)) {
            *abort_flag = 1;
            flag_error(p.dev_err, MOE_DEV_TIMEOUT);
            break;
          }
          const int kb = uu * p.KS;
          const int nq = KB - kb < p.KS ? KB - kb : p.KS;
          uint8_t* sA = base + (size_t)stage * stageBytes;
          const uint32_t tx = (kGateUp ? 2 * kABytes : nq * kABytes) + nq * 2 * (kGateUp ? p.NM : ti.np) * 128;
          tc::mbar_arrive_expect_tx(&full[stage], tx);
          if (p.tiled) {
            const int blk = (ti.ws * MT + ti.m) * KB + kb;
            if (kGateUp || nq == 2)
              tc::tma_load_3d(sA, &tmA0, 0, 0, blk, &full[stage], polA);
            else
              tc::tma_load_3d(sA, &tmA1, 0, 0, blk, &full[stage], polA);
          } else {
            tc::tma_load_3d(sA, &tmA0, kb * kBK, ti.m * kBM, ti.ws, &full[stage], polA);
            if (kGateUp) tc::tma_load_3d(sA + kABytes, &tmA1, kb * kBK, ti.m * kBM, ti.ws, &full[stage], polA);
          }
          if (dep_done) {
            issue_b(t, kb, nq, stage);
          } else {
            pend_t[npend] = t;
            pend_kb[npend] = kb;
            pend_nq[npend] = nq;
            pend_st[npend] = stage;
            ++npend;
          }
          ++n_issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!dep_done) resolve();
      *issued = n_issued;
      if (!kGateUp && p.pf.base && !*abort_flag) l2_prefetch_next_layer(p.pf, p.E, c, gridDim.x);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    tc::griddep_wait();
    if (p.ready_flag) load_partition();
    if (tc::elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      const int nbp = p.NB / kGroup;  // buffer groups
      int pc = 0;               // groups committed (selects the group)
      int pb = 0;               // current group
      uint32_t tphase = 0;      // bit b: phase parity of group b
      int n_consumed = 0;
      bool stop = false;
      Segments sg;
      sg.init(s0, s1, KU, false);
      for (int si = 0; si < sg.n && !stop; ++si) {
        int t, u0, u1;
        sg.get(si, t, u0, u1);
        const Tile ti = tile_info(p, U, t, false);
        if (!ti.ok) continue;
        const uint32_t idesc = idesc_e4m3_f32(kBM, 2 * (kGateUp ? p.NM : ti.np));
        // Groups are kGroup consecutive k-blocks counted from the segment's
        // first k-block; the epilogue walks the same groups.
        const int kb_first = u0 * p.KS;
        const int kb_end = u1 * p.KS < KB ? u1 * p.KS : KB;
        for (int uu = u0; uu < u1 && !stop; ++uu) {
          if (!tc::mbar_wait_bounded(&full[stage], phase, abort_flag, kWaitBudgetNs)) {
            *abort_flag = 1;
            flag_error(p.dev_err, MOE_DEV_TIMEOUT);
            stop = true;
            break;
          }
          tc::tc_fence_after();
          const int nq = KB - uu * p.KS < p.KS ? KB - uu * p.KS : p.KS;
          const uint32_t aAddr = tc::smem_u32(base + (size_t)stage * stageBytes);
          const uint32_t bAddr = aAddr + aBytes;
          for (int q = 0; q < nq; ++q) {
            const int kb = uu * p.KS + q;
            const int half = (kb - kb_first) % kGroup;
            if (half == 0) {
              pb = pc % nbp;
              if (!tc::mbar_wait_bounded(&tempty[pb], ((tphase >> pb) & 1u) ^ 1u, abort_flag, kWaitBudgetNs)) {
                *abort_flag = 1;
                flag_error(p.dev_err, MOE_DEV_TIMEOUT);
                stop = true;
                break;
              }
              tc::tc_fence_after();
            }
            const uint32_t d0 = tmem_base + (kGroup * pb + half) * buf_cols;
            const uint32_t aq = aAddr + (kGateUp ? 0 : q * kABytes);
            const uint32_t bq = bAddr + q * bStride;
#pragma unroll
            for (int kk = 0; kk < kBK / 32; ++kk) {
              const uint32_t accum = kk > 0 ? 1u : 0u;
              const uint64_t bdesc = tc::smem_desc_sw128(bq + kk * 32);
              mma_e4m3(d0, tc::smem_desc_sw128(aq + kk * 32), bdesc, idesc, accum);
              if (kGateUp) mma_e4m3(d0 + 2 * p.NM, tc::smem_desc_sw128(aq + kABytes + kk * 32), bdesc, idesc, accum);
            }
            if (half == kGroup - 1 || kb + 1 == kb_end) {
              tc::mma_commit(&tfull[pb]);
              tphase ^= 1u << pb;
              ++pc;
            }
          }
          if (stop) break;
          tc::mma_commit(&empty[stage]);
          ++n_consumed;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      *consumed = n_consumed;
      tc::mma_commit(drain);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const int etid = threadIdx.x - 64;
    tc::griddep_wait();
    if (p.ready_flag) load_partition();
    if (etid == 0 && blockIdx.x == 0 && U != 0 && !(U >= 1 && U <= p.cap)) flag_error(p.dev_err, MOE_DEV_CAPACITY);
    // down: gate/up has finished, so no CTA still reads the handshake word
    if (!kGateUp && p.ready_clear && etid == 0 && blockIdx.x == 0) *p.ready_clear = 0;
    const int first_tile_c = KU > 0 ? static_cast<int>(s0 / KU) : 0;
    const int KBs = p.K / 128;  // scale blocks along K (== KB)
    const int nbp = p.NB / kGroup;  // TMEM buffer groups
    int pc = 0;                 // groups consumed
    uint32_t tphase = 0;        // bit b: phase parity of group b
    bool stop = false;
    Segments sg;
    sg.init(s0, s1, KU, false);
    for (int si = 0; si < sg.n && !stop; ++si) {
      int t, u0, u1;
      sg.get(si, t, u0, u1);
      const Tile ti = tile_info(p, U, t, true);
      if (!ti.ok) {
        if (etid == 0) flag_error(p.dev_err, MOE_DEV_BAD_ID);
        continue;
      }
      if (!ti.prow_ok && etid == 0) flag_error(p.dev_err, MOE_DEV_BAD_ID);
      // A tile this CTA shares: if every other contributor has already
      // counted in (acquire, read before this segment's k-blocks), this CTA
      // is the last to arrive and can finish the tile at its end without
      // writing its own partials or taking the atomic.
      bool others_done = false;
      if (etid == 0 && !(u0 == 0 && u1 == KU)) {
        const long long t0 = (long long)t * KU;
        const int cf0 = static_cast<int>(seg_owner(t0, total, G));
        const int cl0 = static_cast<int>(seg_owner(t0 + KU - 1, total, G));
        int cnt;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(cnt) : "l"(p.tile_cnt + t) : "memory");
        others_done = cnt == cl0 - cf0;
      }
      // gate/up is token-dense (column n is token n): the expert's tokens as
      // a mask over the columns, a token's rank in it giving its Hq row
      const int nb = kGateUp ? p.NM : ti.np;
      uint32_t mask = 0;
      bool mok = true;
      if (kGateUp) {
        const bool mine = lane < ti.ne;
        const int tok = mine ? p.perm_token[ti.off + lane] : 0;
        const int prev = __shfl_up_sync(0xFFFFFFFFu, tok, 1);
        const bool okk = !mine || (tok >= 0 && tok < p.T && (lane == 0 || tok > prev));
        mask = __reduce_or_sync(0xFFFFFFFFu, (mine && tok >= 0 && tok < 32) ? 1u << tok : 0u);
        mok = __all_sync(0xFFFFFFFFu, okk);
        if (!mok && etid == 0) flag_error(p.dev_err, MOE_DEV_BAD_ID);
      }
      const int row = ti.m * kBM + r;
      const bool row_ok = row < p.M;
      float ga[kMaxNM], ua[kMaxNM];
#pragma unroll
      for (int n = 0; n < kMaxNM; ++n) ga[n] = ua[n] = 0.f;
      // Per-row activation scales of gate/up are constant over the tile.
      const int kb_first = u0 * p.KS;
      const int kb_end = u1 * p.KS < KB ? u1 * p.KS : KB;
      const float* wsg = p.wscale + ((size_t)ti.e * p.scale_rows + ti.m) * KBs;
      const float* wsu = p.wscale + ((size_t)ti.e * p.scale_rows + p.M / 128 + ti.m) * KBs;
      // Row scales of the B operand: per row for gate/up (constant over the
      // tile), per (k-block, row) for down, stored k-block-major so that a
      // tile's rows are contiguous (four 16-byte loads per 16 rows).
      float sbr[kMaxNM];
#pragma unroll
      for (int n = 0; n < kMaxNM; ++n) sbr[n] = 0.f;
      const int prow0 = ti.prow_ok ? ti.prow : 0;
      if (kGateUp) {
#pragma unroll
        for (int cc = 0; cc < kMaxNM / 16; ++cc)
          if (cc < nb / 16) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 v = __ldg(reinterpret_cast<const float4*>(p.bscale + cc * 16 + q * 4));
              sbr[cc * 16 + q * 4] = v.x;
              sbr[cc * 16 + q * 4 + 1] = v.y;
              sbr[cc * 16 + q * 4 + 2] = v.z;
              sbr[cc * 16 + q * 4 + 3] = v.w;
            }
          }
      }
      // Promotes one k-block's buffer: acc += w_scale * s_row * (hi + lo / 16).
      auto promote = [&](uint32_t tb, float sg, float su, const float* sb_row) {
#pragma unroll
        for (int cc = 0; cc < kMaxNM / 16; ++cc) {
          if (cc < nb / 16) {
            float gh[16], gl[16], uh[16], ul[16];
            tc::tmem_ld16(tb + cc * 16, gh);
            tc::tmem_ld16(tb + nb + cc * 16, gl);
            if (kGateUp) {
              tc::tmem_ld16(tb + 2 * p.NM + cc * 16, uh);
              tc::tmem_ld16(tb + 2 * p.NM + nb + cc * 16, ul);
            }
            tc::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int n = cc * 16 + j;
              const float sb = sb_row[n];
              ga[n] = fmaf(sg * sb, fmaf(gl[j], 1.f / kLoScale, gh[j]), ga[n]);
              if (kGateUp) ua[n] = fmaf(su * sb, fmaf(ul[j], 1.f / kLoScale, uh[j]), ua[n]);
            }
          }
        }
      };
      auto load_row_scales = [&](int kb, float* dst) {  // down: per (k-block, row)
        const float* src = p.bscale + (size_t)kb * p.hs_stride + prow0;
#pragma unroll
        for (int cc = 0; cc < kMaxNM / 16; ++cc)
          if (cc < nb / 16) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 v = __ldg(reinterpret_cast<const float4*>(src + cc * 16 + q * 4));
              dst[cc * 16 + q * 4] = v.x;
              dst[cc * 16 + q * 4 + 1] = v.y;
              dst[cc * 16 + q * 4 + 2] = v.z;
              dst[cc * 16 + q * 4 + 3] = v.w;
            }
          }
      };
      for (int kb = kb_first; kb < kb_end; kb += kGroup) {
        const bool two = kGroup == 2 && kb + 1 < kb_end;
        const int pb = pc % nbp;
        // Scales of both k-blocks are requested before waiting for their
        // MMAs, so their latency hides behind the wait.
        const float sg0 = __ldg(&wsg[kb]);
        const float su0 = kGateUp ? __ldg(&wsu[kb]) : 0.f;
        const float sg1 = two ? __ldg(&wsg[kb + 1]) : 0.f;
        const float su1 = kGateUp && two ? __ldg(&wsu[kb + 1]) : 0.f;
        float sbr1[kMaxNM];
        if (!kGateUp) {
          load_row_scales(kb, sbr);
          if (two) load_row_scales(kb + 1, sbr1);
        }
        // Warp-uniform wait: a warp that gives up keeps walking the same
        // loop (skipping the arithmetic) so every later barrier is reached.
        bool ok = tc::mbar_wait_bounded(&tfull[pb], (tphase >> pb) & 1u, abort_flag, kWaitBudgetNs);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok && lane == 0) {
          *abort_flag = 1;
          flag_error(p.dev_err, MOE_DEV_TIMEOUT);
        }
        if (ok) {
          tc::tc_fence_after();
          const uint32_t tb = tmem_base + lane_off + kGroup * pb * buf_cols;
          promote(tb, sg0, su0, sbr);
          if (two) promote(tb + buf_cols, sg1, su1, kGateUp ? sbr : sbr1);
        }
        tc::tc_fence_before();
        tc::mbar_arrive(&tempty[pb]);
        tphase ^= 1u << pb;
        ++pc;
      }
      tc::named_bar_sync(1, kEpiThreads);
      if (*abort_flag) {
        stop = true;
        break;
      }

      const bool whole = u0 == 0 && u1 == KU;
      bool finished = whole;
      if (!whole) {
        const long long t0 = (long long)t * KU;
        const int cf = static_cast<int>(seg_owner(t0, total, G));
        const int cl = static_cast<int>(seg_owner(t0 + KU - 1, total, G));
        if (etid == 0) *bcast = others_done ? -1 : 0;
        tc::named_bar_sync(1, kEpiThreads);
        bool last = *bcast == -1;
        tc::named_bar_sync(1, kEpiThreads);  // bcast is reused below
        if (!last) {
          float* P = p.partials + ((size_t)c * 2 + (t == first_tile_c ? 0 : 1)) * (size_t)(2 * p.NM * 128);
#pragma unroll
          for (int n = 0; n < kMaxNM; ++n) {
            if (n < nb) {
              P[(size_t)n * 128 + r] = ga[n];
              if (kGateUp) P[(size_t)(p.NM + n) * 128 + r] = ua[n];
            }
          }
          tc::named_bar_sync(1, kEpiThreads);
          if (etid == 0) {
            __threadfence();
            *bcast = atomicAdd(&p.tile_cnt[t], 1);
          }
          tc::named_bar_sync(1, kEpiThreads);
          last = *bcast == cl - cf;
          tc::named_bar_sync(1, kEpiThreads);
        }
        if (last) {
          __threadfence();
          finished = true;
          // Sum in CTA order from zero, 16 columns at a time: each other
          // contributor's 16 (gate/up: 32) loads are unconditional, so they
          // are all in flight before the first add; this CTA's own partial
          // is still in registers.
#pragma unroll
          for (int cc = 0; cc < kMaxNM / 16; ++cc) {
            if (cc < nb / 16) {
              float g[16], v[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) g[j] = v[j] = 0.f;
              for (int q2 = cf; q2 <= cl; ++q2) {
                if (q2 == c) {
#pragma unroll
                  for (int j = 0; j < 16; ++j) {
                    g[j] += ga[cc * 16 + j];
                    if (kGateUp) v[j] += ua[cc * 16 + j];
                  }
                } else {
                  const int ft = static_cast<int>((total * q2 / G) / KU);
                  const float* P2 =
                      p.partials + ((size_t)q2 * 2 + (t == ft ? 0 : 1)) * (size_t)(2 * p.NM * 128) + (size_t)cc * 16 * 128 + r;
                  float lg[16], lv[16];
#pragma unroll
                  for (int j = 0; j < 16; ++j) {
                    lg[j] = __ldcg(P2 + (size_t)j * 128);
                    if (kGateUp) lv[j] = __ldcg(P2 + (size_t)(p.NM + j) * 128);
                  }
#pragma unroll
                  for (int j = 0; j < 16; ++j) {
                    g[j] += lg[j];
                    if (kGateUp) v[j] += lv[j];
                  }
                }
              }
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                ga[cc * 16 + j] = g[j];
                ua[cc * 16 + j] = v[j];
              }
            }
          }
        }
      }
      if (!finished) continue;

      if (kGateUp) {
        // h = silu(gate) * up, quantized per (token, 128-row block) for the
        // down projection, with the power-of-two scale of max |h| over the
        // block's rows.
        // Every column of a 16-column chunk is computed (columns of tokens
        // outside the expert's group hold finite values and are dropped at
        // the store), with no per-token branch.  This code runs once per
        // tile, so its instructions are usually not in the SM's instruction
        // cache: it is kept short (one warp max instruction per column,
        // each column's scale computed once by one thread).
        float h[kMaxNM];
#pragma unroll
        for (int cc = 0; cc < kMaxNM / 16; ++cc) {
          if (cc < nb / 16) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int n = cc * 16 + j;
              const float s = silu_mul(ga[n], ua[n]);
              h[n] = (((mask >> n) & 1u) && row_ok) ? s : 0.f;
              // max |h| over the warp's rows; |h| >= 0 orders as its bits,
              // and a NaN counts as 0 (as fmaxf would skip it)
              const float a = fabsf(h[n]);
              const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, a == a ? __float_as_uint(a) : 0u);
              if (lane == 0) s_red[q4 * kMaxNM + n] = __uint_as_float(m);
            }
          }
        }
        tc::named_bar_sync(1, kEpiThreads);
        if (etid < nb) {  // column etid's scale, from the four warps' maxima
          const int n = etid;
          const float amax =
              fmaxf(fmaxf(s_red[n], s_red[kMaxNM + n]), fmaxf(s_red[2 * kMaxNM + n], s_red[3 * kMaxNM + n]));
          float sc, inv_sc;
          pow2_scale(amax, sc, inv_sc);
          s_sc[n] = inv_sc;
          if (((mask >> n) & 1u) && ti.prow_ok && mok)
            p.hscale[(size_t)ti.m * p.hs_stride + ti.prow + __popc(mask & ((1u << n) - 1u))] = sc;
        }
        tc::named_bar_sync(1, kEpiThreads);
#pragma unroll
        for (int cc = 0; cc < kMaxNM / 16; ++cc) {
          if (cc < nb / 16) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int n = cc * 16 + j;
              if (((mask >> n) & 1u) && ti.prow_ok && mok && row_ok) {
                uint8_t hi, lo;
                split_e4m3(h[n] * s_sc[n], hi, lo);
                const int rr = ti.prow + __popc(mask & ((1u << n) - 1u));  // the token's row in the group
                p.hq_hi[(size_t)rr * p.M + row] = hi;
                p.hq_lo[(size_t)rr * p.M + row] = lo;
              }
            }
          }
        }
        tc::named_bar_sync(1, kEpiThreads);  // s_red and s_sc are reused by the next tile
      } else {
#pragma unroll
        for (int n = 0; n < kMaxNM; ++n)
          if (n < ti.ne && row_ok) p.o[(size_t)(ti.off + n) * p.M + row] = ga[n];
      }
    }
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  if (*abort_flag) {
    if (threadIdx.x == 0) {
      for (int i = *consumed; i < *issued; ++i)
        tc::mbar_wait_bounded(&full[i % S], static_cast<uint32_t>((i / S) & 1), nullptr, 100000000ull);
    }
  }
  if (warp == 1) {
    tc::mbar_wait_bounded(drain, 0, nullptr, 100000000ull);
    __syncwarp();
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

// Token-dense prep (standalone calls and layers with an expert pool; in the
// whole step the layer head's extra CTAs do this work): CTA t finds max |x|
// of token row t, quantizes the row once (power-of-two scale, hi/lo E4M3
// pair) into row t of Xq; padding rows up to NM get scale 1 (their operand
// rows read as zeros).  All CTAs zero the fix-up counters.
constexpr int kPrepThreads = 256;

__global__ void __launch_bounds__(kPrepThreads) ffn_fp8_prep_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ x_rows, int x_rows_limit, int T, int NM, int H,
    uint8_t* __restrict__ xq_hi, uint8_t* __restrict__ xq_lo, float* __restrict__ xscale,
    int32_t* __restrict__ counters, int n_counters, int32_t* dev_err) {
  __shared__ float s_max[kPrepThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  for (int i = blockIdx.x * blockDim.x + tid; i < n_counters; i += gridDim.x * blockDim.x) counters[i] = 0;
  for (int t = blockIdx.x; t < NM; t += gridDim.x) {
    const long long row = t < T ? (x_rows ? x_rows[t] : t) : -1;
    const bool ok = t < T && row >= 0 && (!x_rows || row < x_rows_limit);
    if (t < T && !ok && tid == 0) flag_error(dev_err, MOE_DEV_BAD_ID);
    fp8q::quantize_row(ok ? x + (size_t)row * H : nullptr, H, xq_hi + (size_t)t * H, xq_lo + (size_t)t * H,
                       t < T ? xscale + t : nullptr, s_max, t < T);
    if (t >= T && tid == 0) xscale[t] = 1.f;
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool make_tmap_u8(CUtensorMap* tm, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                  const uint32_t* box_dims) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[3], gstride[2];
  cuuint32_t box[3], estr[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    box[i] = box_dims[i];
  }
  for (int i = 0; i < rank - 1; ++i) gstride[i] = strides_bytes[i];
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), gdim, gstride, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Fp8Geom {
  int NM, MT_gu, MT_d, Rh, G, KS_d, stages_gu, stages_d;
  size_t smem_gu, smem_d;
};

constexpr size_t kSmemLimit = 227 * 1024;
constexpr size_t kSmemExtra = 1024 + kBarRegion + 4 * 5 * kMaxNM;

Fp8Geom fp8_geom(const moe_layer_weights& lw, int T, int k) {
  Fp8Geom g;
  const int TK = T * k;
  const int cap = lw.E < TK ? lw.E : TK;
  g.NM = (T + 15) & ~15;
  g.MT_gu = lw.I / kBM;
  g.MT_d = lw.H / kBM;
  g.Rh = cap * g.NM;  // expert u's token rows of the intermediate from u * NM
  g.G = sm_count();
  g.KS_d = lw.layout == MOE_LAYOUT_TILED ? 2 : 1;
  const size_t b = static_cast<size_t>(2 * g.NM) * 128;
  const size_t st_gu = 2 * kABytes + b, st_d = g.KS_d * (kABytes + b);
  g.stages_gu = static_cast<int>((kSmemLimit - kSmemExtra) / st_gu);
  g.stages_d = static_cast<int>((kSmemLimit - kSmemExtra) / st_d);
  // Four stages in flight per CTA: a same-box sweep of the whole step over
  // 3-6 stages for each kernel (bf16 Qwen-like, GPT-OSS-like and batched
  // workloads; FP8 DeepSeek-like) was fastest at four for both the gate/up
  // and the down kernel, 2-3.5% ahead of the deepest ring that fits.
  if (g.stages_gu > 4) g.stages_gu = 4;
  if (g.stages_d > 4) g.stages_d = 4;
  g.smem_gu = g.stages_gu * st_gu + kSmemExtra;
  g.smem_d = g.stages_d * st_d + kSmemExtra;
  return g;
}

// As many promotion buffers as fit in 512 TMEM columns (at most kNBMax), so
// the MMA can run ahead of the epilogue by several k-blocks.
int nb_for(int cols_per_buffer) {
  int nb = 512 / cols_per_buffer;
  return nb > kNBMax ? kNBMax : nb;
}

uint32_t pow2_cols(int c) {
  uint32_t v = 32;
  while (v < static_cast<uint32_t>(c)) v <<= 1;
  return v;
}

struct Fp8Ws {
  uint8_t *xq_hi, *xq_lo, *hq_hi, *hq_lo;
  float *xscale, *hscale, *o, *partials;
  int32_t* counters;
  int n_counters;
  size_t bytes;
};

Fp8Ws fp8_carve(const moe_layer_weights& lw, int T, int k, void* base) {
  Fp8Geom g = fp8_geom(lw, T, k);
  const int TK = T * k;
  const int cap = lw.E < TK ? lw.E : TK;
  char* p0 = static_cast<char*>(base);
  char* p = p0;
  Fp8Ws w;
  auto take = [&](size_t bytes) {
    char* r = p;
    p += align_up(bytes, 256);
    return r;
  };
  w.xq_hi = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(T) * lw.H));
  w.xq_lo = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(T) * lw.H));
  w.xscale = reinterpret_cast<float*>(take(static_cast<size_t>(kMaxNM) * 4));
  w.hq_hi = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(g.Rh) * lw.I));
  w.hq_lo = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(g.Rh) * lw.I));
  w.hscale = reinterpret_cast<float*>(take(static_cast<size_t>(g.Rh) * (lw.I / 128) * 4));
  w.o = reinterpret_cast<float*>(take(static_cast<size_t>(TK) * lw.H * 4));
  w.partials = reinterpret_cast<float*>(take(static_cast<size_t>(g.G) * 2 * 2 * g.NM * 128 * 4));
  w.n_counters = cap * (g.MT_gu + g.MT_d);
  w.counters = reinterpret_cast<int32_t*>(take(static_cast<size_t>(w.n_counters) * 4));
  w.bytes = static_cast<size_t>(p - p0);
  return w;
}

}  // namespace

bool ffn_fp8_supported(const moe_layer_weights& lw, int T, int k) {
  if (lw.dtype != MOE_DTYPE_E4M3_B128) return false;
  if (lw.layout != MOE_LAYOUT_ROWMAJOR && lw.layout != MOE_LAYOUT_TILED) return false;
  if (lw.H % kBK || lw.I % kBK) return false;
  if (T < 1 || T > kMaxNM) return false;
  Fp8Geom g = fp8_geom(lw, T, k);
  return g.stages_gu >= 2 && g.stages_d >= 2 && encode_fn() != nullptr;
}

size_t ffn_fp8_workspace_bytes(const moe_layer_weights& lw, int T, int k) {
  return fp8_carve(lw, T, k, nullptr).bytes;
}

bool ffn_fp8_head_prep(const moe_layer_weights& lw, int T, int k, void* ws, HeadPrep* hp) {
  if (!ffn_fp8_supported(lw, T, k) || lw.pool) return false;
  Fp8Ws w = fp8_carve(lw, T, k, ws);
  hp->xq_hi = w.xq_hi;
  hp->xq_lo = w.xq_lo;
  hp->xscale = w.xscale;
  hp->q_rows = fp8_geom(lw, T, k).NM;
  hp->counters = w.counters;
  hp->n_counters = w.n_counters;
  hp->H = lw.H;
  return true;
}

int ffn_fp8_launch(const FfnArgs& a) {
  const auto& lw = a.lw;
  const int T = a.T, k = a.k, TK = T * k;
  const int cap = lw.E < TK ? lw.E : TK;
  Fp8Geom g = fp8_geom(lw, T, k);
  Fp8Ws ws = fp8_carve(lw, T, k, a.ws);
  int32_t* cnt_gu = ws.counters;
  int32_t* cnt_d = cnt_gu + static_cast<size_t>(cap) * g.MT_gu;

  const uint64_t H = lw.H, I = lw.I, E = weight_slots(lw);  // E: expert slots in the buffers
  const uint64_t KBg = H / kBK, KBd = I / kBK;
  CUtensorMap tm_g, tm_u, tm_xh, tm_xl, tm_wd, tm_wd1, tm_hh, tm_hl;
  if (lw.layout == MOE_LAYOUT_TILED) {
    {
      uint64_t dims[3] = {kBK, 2 * kBM, E * g.MT_gu * KBg}, str[2] = {kBK, 2 * kABytes};
      uint32_t box[3] = {kBK, 2 * kBM, 1};
      if (!make_tmap_u8(&tm_g, lw.w_gate_up, 3, dims, str, box)) return MOE_ERR_CUDA;
      tm_u = tm_g;
    }
    {
      uint64_t dims[3] = {kBK, kBM, E * g.MT_d * KBd}, str[2] = {kBK, kABytes};
      uint32_t box2[3] = {kBK, kBM, 2}, box1[3] = {kBK, kBM, 1};
      if (!make_tmap_u8(&tm_wd, lw.w_down, 3, dims, str, box2)) return MOE_ERR_CUDA;
      if (!make_tmap_u8(&tm_wd1, lw.w_down, 3, dims, str, box1)) return MOE_ERR_CUDA;
    }
  } else {
    uint32_t box[3] = {kBK, kBM, 1};
    {
      uint64_t dims[3] = {H, I, E}, str[2] = {H, 2 * I * H};
      if (!make_tmap_u8(&tm_g, lw.w_gate_up, 3, dims, str, box)) return MOE_ERR_CUDA;
      const char* up = static_cast<const char*>(lw.w_gate_up) + I * H;
      if (!make_tmap_u8(&tm_u, up, 3, dims, str, box)) return MOE_ERR_CUDA;
    }
    {
      uint64_t dims[3] = {I, H, E}, str[2] = {I, H * I};
      if (!make_tmap_u8(&tm_wd, lw.w_down, 3, dims, str, box)) return MOE_ERR_CUDA;
      tm_wd1 = tm_wd;
    }
  }
  {
    // the T quantized token rows; the box's rows past T read as zeros
    uint64_t dims[2] = {H, static_cast<uint64_t>(T)}, str[1] = {H};
    uint32_t box[2] = {kBK, static_cast<uint32_t>(g.NM)};
    if (!make_tmap_u8(&tm_xh, ws.xq_hi, 2, dims, str, box)) return MOE_ERR_CUDA;
    if (!make_tmap_u8(&tm_xl, ws.xq_lo, 2, dims, str, box)) return MOE_ERR_CUDA;
  }
  {
    uint64_t dims[2] = {I, static_cast<uint64_t>(g.Rh)}, str[1] = {I};
    uint32_t box[2] = {kBK, 16};
    if (!make_tmap_u8(&tm_hh, ws.hq_hi, 2, dims, str, box)) return MOE_ERR_CUDA;
    if (!make_tmap_u8(&tm_hl, ws.hq_lo, 2, dims, str, box)) return MOE_ERR_CUDA;
  }

  cudaStream_t s = a.stream;
  if (!a.head_prepared) {
    LaunchScope ls(kProfPrep, s);
    if (launch_k(ffn_fp8_prep_kernel, dim3(g.NM), dim3(kPrepThreads), 0, s, a.pdl_first,
                 static_cast<const uint16_t*>(a.x), a.x_rows, a.x_rows_limit, T, g.NM, lw.H, ws.xq_hi, ws.xq_lo,
                 ws.xscale, ws.counters, ws.n_counters, a.dev_err) != MOE_OK)
      return MOE_ERR_CUDA;
  }

  Fp8Params fp{};
  fp.T = T;
  fp.k = k;
  fp.E = lw.E;
  fp.cap = cap;
  fp.NM = g.NM;
  fp.Rh = g.Rh;
  fp.hs_stride = g.Rh;
  fp.tiled = lw.layout == MOE_LAYOUT_TILED ? 1 : 0;
  fp.pdl = 1;
  fp.n_unique = a.n_unique;
  fp.unique = a.unique;
  fp.offsets = a.offsets;
  fp.perm_token = a.perm_token;
  fp.ready_flag = a.head_prepared ? a.ready_flag : nullptr;
  fp.ready_value = a.ready_value;
  fp.hq_hi = ws.hq_hi;
  fp.hq_lo = ws.hq_lo;
  fp.hscale = ws.hscale;
  fp.o = ws.o;
  fp.partials = ws.partials;
  fp.dev_err = a.dev_err;
  fp.slot_of = slot_table(lw);
  fp.n_slots = weight_slots(lw);

  // gate/up
  fp.M = lw.I;
  fp.K = lw.H;
  fp.KS = 1;
  fp.stages = g.stages_gu;
  fp.NB = nb_for(4 * g.NM);
  fp.tmem_cols = pow2_cols(fp.NB * 4 * g.NM);
  fp.wscale = lw.scales_gate_up;
  fp.scale_rows = 2 * lw.I / 128;
  fp.bscale = ws.xscale;
  fp.tile_cnt = cnt_gu;
  if (cudaFuncSetAttribute(ffn_fp8_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(g.smem_gu)) != cudaSuccess)
    return MOE_ERR_CUDA;
  {
    LaunchScope ls(kProfGateUp, s);
    if (launch_k(ffn_fp8_kernel<true>, dim3(g.G), dim3(kThreads), g.smem_gu, s, true, tm_g, tm_u, tm_xh, tm_xl,
                 fp) != MOE_OK)
      return MOE_ERR_CUDA;
  }
  // down + combine
  fp.pf = a.pf;
  fp.M = lw.H;
  fp.K = lw.I;
  fp.KS = g.KS_d;
  fp.stages = g.stages_d;
  fp.NB = nb_for(2 * g.NM);
  fp.tmem_cols = pow2_cols(fp.NB * 2 * g.NM);
  fp.wscale = lw.scales_down;
  fp.scale_rows = lw.H / 128;
  fp.bscale = ws.hscale;
  fp.tile_cnt = cnt_d;
  fp.ready_clear = fp.ready_flag;
  fp.ready_flag = nullptr;
  if (cudaFuncSetAttribute(ffn_fp8_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(g.smem_d)) != cudaSuccess)
    return MOE_ERR_CUDA;
  {
    LaunchScope ls(kProfDown, s);
    if (launch_k(ffn_fp8_kernel<false>, dim3(g.G), dim3(kThreads), g.smem_d, s, true, tm_wd, tm_wd1, tm_hh, tm_hl,
                 fp) != MOE_OK)
      return MOE_ERR_CUDA;
  }
  // Weighted combine of the per-(token, slot) outputs, slot order.
  return combine_launch(a, ws.o, true);
}

}  // namespace moe
