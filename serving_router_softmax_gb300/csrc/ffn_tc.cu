// moe_verify_ffn, tensor-core path (bf16 weights): TMA-streamed expert weights
// feeding tcgen05 MMAs with fp32 accumulators in TMEM.
//
// The verify step's MoE cost is the union of the experts its tokens activate
// (EcoSpec write-up, sections 1-2); this path reads each unique expert's
// weights from HBM exactly once and applies them to all of that expert's
// tokens.  Per layer:
//   prep     padded per-expert token groups: gathers x rows into Xp (each
//            expert's group starts on a 16-row boundary, pad rows zeroed),
//            zeroes the fixup counters.
//   gate/up  h = silu(W_gate x) * (W_up x) for every (expert, token) pair,
//            written as bf16 into Hp (same padded rows).
//   down     o = W_down h, then y_t = sum_j w_tj o_(t,j) in slot order.
//
// Tiling: a tile is 128 weight rows of one expert (the MMA's M) times all of
// that expert's tokens (N = group size rounded up to 16, at most 256); K is
// streamed in 64-element (128-byte) blocks through a TMA -> shared memory ring.
// The weights are the A operand, the tokens the B operand, both K-major with
// the 128-byte swizzle.  The skinny N makes the kernels HBM-bound; tensor
// cores only keep the arithmetic off the critical path.
//
// Load balance: the number of unique experts is only known on the device, so
// the grid is persistent (one CTA per SM) and splits the layer's k-blocks
// evenly (stream-K).  A tile cut between CTAs is finished by the last CTA to
// arrive (atomic counter, no waiting), which sums the fp32 partials of all
// contributors in CTA order, so results do not depend on timing.  The down
// weighted combine is its own kernel afterwards.
//
// Roles per CTA (192 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues MMAs, warps 2-5 drain accumulators (TMEM lane quarter = warp % 4).
// Every wait on an mbarrier is bounded; on time-out the CTA raises
// MOE_DEV_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM and exits.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "ffn_internal.cuh"
#include "tc_ptx.cuh"
#include "stream_k.cuh"
#include "l2_prefetch.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;          // weight rows per tile (MMA M)
constexpr int kBK = 64;           // K elements per stage (128 bytes of bf16)
constexpr int kABytes = kBM * kBK * 2;
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint64_t kWaitBudgetNs = 2000000000ull;  // 2 s
constexpr uint64_t kReadyBudgetNs = 100000ull;     // 100 us for the union handshake
constexpr int kBarRegion = 512;   // mbarriers + flags of the CTA
static_assert((2 * 12 + 5) * 8 + 5 * 4 <= kBarRegion, "barrier region too small");

struct TcParams {
  int T, k, E, cap;
  int M, K;          // rows of each expert matrix, reduction length
  int NM;            // max padded token columns (multiple of 16, <= 256)
  int Rmax;          // rows of Xp
  int Rh;            // rows of Hp
  int dense;         // token-dense gate/up (see ffn_tc_dense)
  int tiled;         // weights in the tile-packed layout (else row-major)
  int tail_rows;     // tiled: rows loaded for the last M-tile when M % 128 leaves it
                     // partly padding (multiple of 8, < 128), else 0
  int KS;            // k-blocks per pipeline stage (1, or 2 for tiled down)
  int stages;
  int pdl;           // launched with programmatic dependent launch
  int stall;         // test hook: the producer issues nothing, so the bounded waits run out
  int acc_stages;
  uint32_t tmem_cols;
  const int32_t* n_unique;
  const int32_t* unique;
  const int32_t* offsets;
  const int32_t* perm_token;
  const int32_t* poff;
  uint16_t* hp;      // gate/up output, [R_pad_max][M] bf16
  float* o;          // down output, [T*k][M] fp32 (perm order)
  float* partials;   // [grid][2][2*NM][128] fp32
  int32_t* tile_cnt; // [cap * MT]
  int32_t* dev_err;
  // Union-ready handshake with the layer-head kernel that gate/up follows
  // directly (NULL: a prep kernel sits between them and the union is
  // complete before gate/up starts).  gate/up waits (bounded) until the head
  // has published ready_value in the low 16 bits of ready_flag (the union
  // size in the high bits) before reading the union ahead of its dependency
  // wait.  down (whose union is always complete before it
  // starts) clears ready_clear once gate/up has finished.
  int32_t* ready_flag;
  int32_t ready_value;
  int32_t* ready_clear;
  const int32_t* slot_of;  // expert -> weight slot (NULL: identity)
  int n_slots;
  // down only: the next layer's predicted experts, which each CTA asks L2
  // to fetch (its round-robin share) once it has issued its last weight load.
  NextLayerPrefetch pf;
};

struct Tile {
  int u, m, e, ws, ne, np, prow, off;  // ws: the expert's slot in the weight buffers
  bool ok, prow_ok;
};


__device__ __forceinline__ Tile tile_info(const TcParams& p, int U, int t) {
  Tile ti;
  ti.m = t / U;
  ti.u = t - ti.m * U;
  ti.e = p.unique[ti.u];
  ti.off = p.offsets[ti.u];
  ti.ne = p.offsets[ti.u + 1] - ti.off;
  ti.np = (ti.ne + 15) & ~15;
  ti.prow = p.dense ? ti.u * p.NM : p.poff[ti.u];
  ti.ok = ti.e >= 0 && ti.e < p.E && ti.ne >= 1 && ti.ne <= p.T && ti.np <= p.NM && ti.off >= 0 &&
          ti.off + ti.ne <= p.T * p.k;
  ti.ws = ti.ok ? weight_slot(p.slot_of, p.n_slots, ti.e) : -1;
  ti.ok = ti.ok && ti.ws >= 0;
  ti.prow_ok = ti.prow >= 0 && ti.prow + ti.np <= p.Rh;
  return ti;
}

// The part of tile_info that does not depend on the padded group offsets
// (written by the kernel that runs just before gate/up).  In the token-dense
// gate/up every tile's B operand is the same NM rows, so np is NM there.
__device__ __forceinline__ Tile tile_core(const TcParams& p, int U, int t) {
  Tile ti;
  ti.m = t / U;
  ti.u = t - ti.m * U;
  ti.e = p.unique[ti.u];
  ti.off = p.offsets[ti.u];
  ti.ne = p.offsets[ti.u + 1] - ti.off;
  ti.np = (ti.ne + 15) & ~15;
  ti.prow = -1;
  ti.ok = ti.e >= 0 && ti.e < p.E && ti.ne >= 1 && ti.ne <= p.T && ti.np <= p.NM && ti.off >= 0 &&
          ti.off + ti.ne <= p.T * p.k;
  ti.ws = ti.ok ? weight_slot(p.slot_of, p.n_slots, ti.e) : -1;
  ti.ok = ti.ok && ti.ws >= 0;
  ti.prow_ok = false;
  return ti;
}

// silu(a) * b with the fast exponential and division (relative error near
// 1e-6, below the bf16 rounding of h that follows); it sits in the tile end,
// which runs once per tile and is kept short for that reason.
__device__ __forceinline__ float silu_mul(float a, float b) { return __fdividef(a, 1.f + __expf(-a)) * b; }

// Tokens of a tile's expert as a bit mask over the T <= 32 token columns.
// The group lists its tokens in ascending order (the union's layout), so a
// token's row in the expert's Hp block is the number of its group's tokens
// below it.  All 32 lanes of a warp take part (ne <= T <= 32): lane r reads
// the group's r-th token (group_token, issued before the accumulator wait so
// that the load overlaps it), then group_mask combines the lanes.  Returns
// false for a group that is not strictly ascending or names a token outside
// [0, T).
__device__ __forceinline__ int group_token(const TcParams& p, const Tile& ti, int lane) {
  return lane < ti.ne ? p.perm_token[ti.off + lane] : 0;
}

__device__ __forceinline__ bool group_mask(const TcParams& p, const Tile& ti, int lane, int tok, uint32_t& mask) {
  const bool mine = lane < ti.ne;
  const int prev = __shfl_up_sync(0xFFFFFFFFu, tok, 1);
  const bool ok = !mine || (tok >= 0 && tok < p.T && (lane == 0 || tok > prev));
  mask = __reduce_or_sync(0xFFFFFFFFu, (mine && tok >= 0 && tok < 32) ? 1u << tok : 0u);
  return __all_sync(0xFFFFFFFFu, ok);
}

template <bool kGateUp>
__global__ void __launch_bounds__(kThreads, 1)
    ffn_tc_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                  const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmT,
                  const TcParams p) {
  constexpr int nA = kGateUp ? 2 : 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int aBytes = kGateUp ? 2 * kABytes : p.KS * kABytes;
  const int bStride = p.NM * 128;  // one k-block of B
  const int stageBytes = aBytes + p.KS * bStride;
  const int S = p.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + (size_t)S * stageBytes);
  uint64_t* empty = full + S;
  uint64_t* accf = empty + S;
  uint64_t* acce = accf + 2;
  uint64_t* drain = acce + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* bcast = abort_flag + 1;
  volatile int* issued = bcast + 1;
  volatile int* consumed = issued + 1;
  // Barrier/flag block (at most 2*12 + 9 mbarriers + 5 words) then the combine's staging.

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&accf[a], 1);
      tc::mbar_init(&acce[a], kEpiThreads);
    }
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    *issued = 0;
    *consumed = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&tmA0);
    if (kGateUp) tc::tma_prefetch_desc(&tmA1);
    if (p.tail_rows) tc::tma_prefetch_desc(&tmT);
    tc::tma_prefetch_desc(&tmB);
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
  const int KU = (KB + p.KS - 1) / p.KS;  // pipeline units (stages) per tile
  const int c = blockIdx.x;
  const int acc_cols = nA * p.NM;
  int U = 0, G = 0;
  long long total = 0, s0 = 0, s1 = 0;
  // Reads the union size and partitions the layer's pipeline units over at
  // most `total` CTAs, so that every range is non-empty and the CTAs sharing
  // a tile are exactly the consecutive owners of its k-blocks.  Each role
  // calls it once the union is visible to it.
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

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Under programmatic dependent launch the weights of the first S stages
    // are requested before the previous kernel has finished.  They depend
    // only on the expert union, its slot table and staged weights, all written
    // before the prep kernel's own griddepcontrol.wait returned (prep starts
    // this grid only after that wait); their token operand follows once
    // griddepcontrol.wait returns here.
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
        // The union comes from the kernel this grid follows directly: read
        // it early only once the head has published it (acquire), else
        // (bounded wait ran out) after the dependency wait.
        // The head publishes the union size with it (bits 16..31), which
        // saves one dependent read before the first weight load.
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
        if (kGateUp && p.dense) {
          // all NM token rows in one box; rows past T are filled with zeros
          for (int q = 0; q < nq; ++q) tc::tma_load_2d(sB + q * bStride, &tmB, (kb + q) * kBK, 0, &full[st], polB);
          return;
        }
        const Tile ti = tile_info(p, U, t);
        const int prow = ti.prow_ok ? ti.prow : 0;  // bad offsets: load something in bounds, epilogue skips
        for (int q = 0; q < nq; ++q)
          for (int j = 0; j < ti.np / 16; ++j)
            tc::tma_load_2d(sB + q * bStride + j * 2048, &tmB, (kb + q) * kBK, prow + 16 * j, &full[st], polB);
      };
      auto resolve = [&]() {
        tc::griddep_wait();
        tc::griddep_launch_dependents();
        for (int i = 0; i < npend; ++i) issue_b(pend_t[i], pend_kb[i], pend_nq[i], pend_st[i]);
        npend = 0;
        dep_done = true;
      };
      Segments sg;
      sg.init(s0, s1, KU, true);
      for (int si = p.stall ? sg.n : 0; si < sg.n && !*abort_flag; ++si) {
        int t, u0, u1;
        sg.get(si, t, u0, u1);
        const Tile ti = tile_core(p, U, t);
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
          const int nb = (kGateUp && p.dense) ? p.NM : ti.np;  // B rows
          // The last M-tile of a matrix whose rows stop short of it reads only
          // its real rows (the tile-packed layout stores the rest as zeros);
          // the MMA still runs 128 rows and the epilogue drops rows past M.
          const bool tail = p.tiled && p.tail_rows && ti.m == MT - 1;
          const int a_rows = tail ? p.tail_rows : kBM;
          const uint32_t tx = (kGateUp ? 2 : nq) * a_rows * 128 + nq * nb * 128;
          tc::mbar_arrive_expect_tx(&full[stage], tx);
          if (p.tiled) {
            // Tile-packed weights: block (e, m, kb) is contiguous.  gate/up:
            // one 256-row box holds the gate tile then the up tile; down: one
            // box of nq consecutive 16 KB k-blocks.
            const int blk = (ti.ws * MT + ti.m) * KB + kb;
            if (tail) {
              if (kGateUp) {
                tc::tma_load_3d(sA, &tmT, 0, 0, blk, &full[stage], polA);
                tc::tma_load_3d(sA + kABytes, &tmT, 0, kBM, blk, &full[stage], polA);
              } else {
                for (int q = 0; q < nq; ++q)
                  tc::tma_load_3d(sA + q * kABytes, &tmT, 0, 0, blk + q, &full[stage], polA);
              }
            } else if (kGateUp || nq == 2)
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
      int acc = 0;
      uint32_t acc_phase[2] = {0, 0};
      int n_consumed = 0;
      bool stop = false;
      Segments sg;
      sg.init(s0, s1, KU, true);
      for (int si = 0; si < sg.n && !stop; ++si) {
        int t, u0, u1;
        sg.get(si, t, u0, u1);
        const Tile ti = tile_core(p, U, t);
        if (!ti.ok) continue;
        if (!tc::mbar_wait_bounded(&acce[acc], acc_phase[acc] ^ 1u, abort_flag, kWaitBudgetNs)) {
          *abort_flag = 1;
          flag_error(p.dev_err, MOE_DEV_TIMEOUT);
          break;
        }
        tc::tc_fence_after();
        const uint32_t d0 = tmem_base + acc * acc_cols;
        const uint32_t idesc = tc::idesc_bf16_f32(kBM, (kGateUp && p.dense) ? p.NM : ti.np);
        for (int uu = u0; uu < u1; ++uu) {
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
            // gate/up: A = gate tile, A + 16 KB = up tile; down: k-block q at A + q * 16 KB.
            const uint32_t aq = aAddr + (kGateUp ? 0 : q * kABytes);
            const uint32_t bq = bAddr + q * bStride;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              const uint32_t accum = (uu > u0 || q > 0 || kk > 0) ? 1u : 0u;
              const uint64_t bdesc = tc::smem_desc_sw128(bq + kk * 32);
              tc::mma_bf16(d0, tc::smem_desc_sw128(aq + kk * 32), bdesc, idesc, accum);
              if (kGateUp)
                tc::mma_bf16(d0 + p.NM, tc::smem_desc_sw128(aq + kABytes + kk * 32), bdesc, idesc, accum);
            }
          }
          tc::mma_commit(&empty[stage]);
          ++n_consumed;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (stop) break;
        tc::mma_commit(&accf[acc]);
        acc_phase[acc] ^= 1u;
        if (p.acc_stages == 2) acc ^= 1;
      }
      *consumed = n_consumed;
      // All MMAs issued by this thread complete before the drain barrier flips.
      tc::mma_commit(drain);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int r = q * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int etid = threadIdx.x - 64;  // 0..127
    tc::griddep_wait();
    if (p.ready_flag) load_partition();
    if (etid == 0 && blockIdx.x == 0 && U != 0 && !(U >= 1 && U <= p.cap)) flag_error(p.dev_err, MOE_DEV_CAPACITY);
    // down: gate/up has finished, so no CTA still reads the handshake word
    if (!kGateUp && p.ready_clear && etid == 0 && blockIdx.x == 0) *p.ready_clear = 0;
    int acc = 0;
    uint32_t acc_phase[2] = {0, 0};
    const int first_tile_c = KU > 0 ? static_cast<int>(s0 / KU) : 0;
    Segments sg;
    sg.init(s0, s1, KU, true);
    for (int si = 0; si < sg.n; ++si) {
      int t, u0, u1;
      sg.get(si, t, u0, u1);
      const Tile ti = tile_info(p, U, t);
      if (!ti.ok) {
        if (etid == 0) flag_error(p.dev_err, MOE_DEV_BAD_ID);
        continue;
      }
      if (kGateUp && !ti.prow_ok && etid == 0) flag_error(p.dev_err, MOE_DEV_BAD_ID);
      const int gtok = (kGateUp && p.dense) ? group_token(p, ti, lane) : 0;
      // A tile this CTA shares: if every other contributor has already
      // counted in (acquire, read before waiting for this tile's
      // accumulator), this CTA is the last to arrive and finishes the tile
      // without writing its own partials or taking the atomic.
      bool others_done = false;
      if (etid == 0 && !(u0 == 0 && u1 == KU)) {
        const long long t0 = (long long)t * KU;
        const int cf0 = static_cast<int>(seg_owner(t0, total, G));
        const int cl0 = static_cast<int>(seg_owner(t0 + KU - 1, total, G));
        int cnt;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(cnt) : "l"(p.tile_cnt + t) : "memory");
        others_done = cnt == cl0 - cf0;
      }
      // Every epilogue thread waits; the outcome is made uniform through a
      // shared vote so that no thread is left behind at a named barrier.
      if (!tc::mbar_wait_bounded(&accf[acc], acc_phase[acc], abort_flag, kWaitBudgetNs)) {
        *abort_flag = 1;
        flag_error(p.dev_err, MOE_DEV_TIMEOUT);
      }
      if (etid == 0) *bcast = others_done ? -1 : 0;
      tc::named_bar_sync(1, kEpiThreads);
      const bool early_last = *bcast == -1;
      if (*abort_flag) break;
      tc::tc_fence_after();
      uint32_t mask = 0;
      bool hp_ok = ti.prow_ok;
      if (kGateUp && p.dense) {
        const bool mok = group_mask(p, ti, lane, gtok, mask);
        if (!mok && etid == 0) flag_error(p.dev_err, MOE_DEV_BAD_ID);
        hp_ok = hp_ok && mok;
      }
      const bool whole = u0 == 0 && u1 == KU;
      int cf = c, cl = c;  // the CTAs that share the tile
      const int row = ti.m * kBM + r;
      const bool row_ok = row < p.M;
      const uint32_t tacc = tmem_base + lane_off + acc * acc_cols;
      float* P = p.partials + ((size_t)c * 2 + (t == first_tile_c ? 0 : 1)) * (size_t)(2 * p.NM * 128);
      // Result column n: gate/up writes h to Hp (token-dense: column n is
      // token n, stored at its rank in the expert's group), down writes o.
      auto put = [&](int n, float gv, float vv) {
        if (kGateUp) {
          const bool keep = p.dense ? (n < 32 && ((mask >> n) & 1u)) : n < ti.ne;
          const int rr = ti.prow + (p.dense ? __popc(mask & ((1u << n) - 1u)) : n);
          if (row_ok && hp_ok && keep) p.hp[(size_t)rr * p.M + row] = float_to_bf16_bits_rn(silu_mul(gv, vv));
        } else if (row_ok && n < ti.ne) {
          p.o[(size_t)(ti.off + n) * p.M + row] = gv;
        }
      };
      const int ncols = (kGateUp && p.dense) ? p.NM : ti.np;
      bool finished = whole;
      if (!whole && early_last) {
        const long long t0 = (long long)t * KU;
        cf = static_cast<int>(seg_owner(t0, total, G));
        cl = static_cast<int>(seg_owner(t0 + KU - 1, total, G));
        finished = true;
        __threadfence();
      } else if (!whole) {
        // Split tile: this CTA's sums go to its partial slot first.
        for (int cc = 0; cc < ncols / 16; ++cc) {
          float g[16], v[16];
          tc::tmem_ld16(tacc + cc * 16, g);
          if (kGateUp) tc::tmem_ld16(tacc + p.NM + cc * 16, v);
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            P[(size_t)(cc * 16 + j) * 128 + r] = g[j];
            if (kGateUp) P[(size_t)(p.NM + cc * 16 + j) * 128 + r] = v[j];
          }
        }
        // Last-arriver fixup across the CTAs that share this tile.  The CTA
        // barrier orders every thread's partial stores before thread 0's
        // fence and atomic (release); the finisher fences after observing
        // the count (acquire) before reading the other CTAs' partials.
        tc::named_bar_sync(1, kEpiThreads);
        if (etid == 0) {
          __threadfence();
          *bcast = atomicAdd(&p.tile_cnt[t], 1);
        }
        tc::named_bar_sync(1, kEpiThreads);
        const int arrived = *bcast;
        const long long t0 = (long long)t * KU;
        cf = static_cast<int>(seg_owner(t0, total, G));
        cl = static_cast<int>(seg_owner(t0 + KU - 1, total, G));
        tc::named_bar_sync(1, kEpiThreads);
        finished = arrived == cl - cf;
        if (finished) __threadfence();
      }
      if (finished) {
        // One copy of the result code for whole and fixed-up tiles: it runs
        // once per tile, mostly from a cold instruction cache.  Sums run in
        // CTA order; this CTA's own share is still in the accumulator.  A
        // whole tile starts from -0 (x + -0 == x for every x), a fixed-up
        // one from +0.
        for (int cc = 0; cc < ncols / 16; ++cc) {
          float g[16], v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) g[j] = v[j] = whole ? -0.f : 0.f;
          for (int q2 = cf; q2 <= cl; ++q2) {
            float lg[16], lv[16];
            if (q2 == c) {
              tc::tmem_ld16(tacc + cc * 16, lg);
              if (kGateUp) tc::tmem_ld16(tacc + p.NM + cc * 16, lv);
              tc::tmem_ld_wait();
            } else {
              const int ft = static_cast<int>((total * q2 / G) / KU);
              const float* P2 = p.partials + ((size_t)q2 * 2 + (t == ft ? 0 : 1)) * (size_t)(2 * p.NM * 128) +
                                (size_t)cc * 16 * 128 + r;
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                lg[j] = __ldcg(P2 + (size_t)j * 128);
                if (kGateUp) lv[j] = __ldcg(P2 + (size_t)(p.NM + j) * 128);
              }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              g[j] += lg[j];
              if (kGateUp) v[j] += lv[j];
            }
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) put(cc * 16 + j, g[j], kGateUp ? v[j] : 0.f);
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&acce[acc]);
      acc_phase[acc] ^= 1u;
      if (p.acc_stages == 2) acc ^= 1;
    }
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  if (*abort_flag) {
    // Drain: wait (bounded) for issued-but-unconsumed copies and for every
    // issued MMA before the shared memory and TMEM are given back.
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

// Builds Xp (padded token groups), poff and zeroes the fixup counters.
__global__ void __launch_bounds__(256) ffn_prep_kernel(const uint16_t* __restrict__ x,
                                                       const int32_t* __restrict__ x_rows,
                                                       int x_rows_limit, int T, int k, int H, int cap,
                                                       const int32_t* __restrict__ n_unique,
                                                       const int32_t* __restrict__ offsets,
                                                       const int32_t* __restrict__ perm_token,
                                                       uint16_t* __restrict__ xp, int32_t* __restrict__ poff,
                                                       int32_t* __restrict__ counters, int n_counters,
                                                       float* __restrict__ y, int32_t* dev_err) {
  __shared__ int32_t spoff[1025];
  __shared__ int32_t soff[1025];  // offsets[0..U], for the group searches
  __shared__ int s_bad;
  pdl_wait();
  pdl_trigger();
  const int TK = T * k;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_counters; i += gridDim.x * blockDim.x)
    counters[i] = 0;
  int U = *n_unique;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  if (U < 1 || U > cap) {
    // No usable union (the union call flagged why, or U is out of range):
    // y is defined as zero.
    if (U != 0 && blockIdx.x == 0 && threadIdx.x == 0) flag_error(dev_err, MOE_DEV_CAPACITY);
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < (long long)T * H;
         i += (long long)gridDim.x * blockDim.x)
      y[i] = 0.f;
    return;
  }
  // Padded group starts: warp 0 scans ceil16(n_e) over u.
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (U + 31) / 32;
    const int u0 = lane * per;
    int sum = 0;
    for (int u = u0; u < u0 + per && u < U; ++u) {
      const int a = offsets[u], b = offsets[u + 1];
      if (a < 0 || b > TK || b - a < 1 || b - a > T) s_bad = 1;
      sum += ((b - a) + 15) & ~15;
      soff[u] = a;
    }
    int ex = warp_inclusive_sum(sum, lane);
    ex -= sum;
    for (int u = u0; u < u0 + per && u < U; ++u) {
      spoff[u] = ex;
      ex += ((offsets[u + 1] - offsets[u]) + 15) & ~15;
    }
    if (lane == 31) {
      spoff[U] = ex;
      soff[U] = offsets[U];
      if (offsets[U] != TK || offsets[0] != 0) s_bad = 1;
    }
  }
  __syncthreads();
  if (s_bad) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag_error(dev_err, MOE_DEV_BAD_ID);
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < (long long)T * H;
         i += (long long)gridDim.x * blockDim.x)
      y[i] = 0.f;
    return;
  }
  if (blockIdx.x == 0)
    for (int u = threadIdx.x; u <= U; u += blockDim.x) poff[u] = spoff[u];
  // Gather the real token rows only (one 16-byte chunk per thread-iteration).
  // Pad rows of a group are left as they are: a pad row of the B operand only
  // feeds accumulator columns the epilogue never stores.
  const int TKn = soff[U];
  const int cpr = H / 8;  // chunks per row
  const long long chunks = (long long)TKn * cpr;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < chunks;
       i += (long long)gridDim.x * blockDim.x) {
    const int pp = static_cast<int>(i / cpr);  // perm position
    const int ch = static_cast<int>(i - (long long)pp * cpr);
    // group of perm position pp: largest u with offsets[u] <= pp
    int lo = 0, hi = U - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (soff[mid] <= pp) lo = mid;
      else hi = mid - 1;
    }
    const int rr = spoff[lo] + (pp - soff[lo]);
    const int tok = perm_token[pp];
    bool ok = tok >= 0 && tok < T;
    int row = tok;
    if (ok && x_rows) {
      row = x_rows[tok];
      ok = row >= 0 && row < x_rows_limit;
    }
    if (ok)
      *reinterpret_cast<uint4*>(xp + (size_t)rr * H + ch * 8) =
          *reinterpret_cast<const uint4*>(x + (size_t)row * H + ch * 8);
    else
      flag_error(dev_err, MOE_DEV_BAD_ID);
  }
}

// Token-dense prep (T <= 32): copies the T token rows into Xp rows 0..T-1 and
// zeroes the fix-up counters.  Neither depends on the union; the work still
// follows the wait, so that it never competes with the latency-bound head
// kernel it follows, and it hides behind the gate/up kernel's first weight
// loads (that grid starts at this one's trigger).
__global__ void __launch_bounds__(256) ffn_prep_dense_kernel(const uint16_t* __restrict__ x,
                                                             const int32_t* __restrict__ x_rows,
                                                             int x_rows_limit, int T, int H,
                                                             uint16_t* __restrict__ xp,
                                                             int32_t* __restrict__ counters, int n_counters,
                                                             int32_t* dev_err) {
  pdl_wait();
  pdl_trigger();
  const long long tid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long nth = (long long)gridDim.x * blockDim.x;
  for (long long i = tid; i < n_counters; i += nth) counters[i] = 0;
  const int cpr = H / 8;  // 16-byte chunks per row
  for (long long i = tid; i < (long long)T * cpr; i += nth) {
    const int t = static_cast<int>(i / cpr);
    const int ch = static_cast<int>(i - (long long)t * cpr);
    const long long row = x_rows ? x_rows[t] : t;
    if (row >= 0 && (!x_rows || row < x_rows_limit))
      *reinterpret_cast<uint4*>(xp + (size_t)t * H + ch * 8) =
          *reinterpret_cast<const uint4*>(x + (size_t)row * H + ch * 8);
    else
      flag_error(dev_err, MOE_DEV_BAD_ID);
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

// bf16 tensor map with the 128-byte swizzle; dims/box innermost first.
bool make_tmap(CUtensorMap* tm, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
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
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), gdim, gstride, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct TcGeom {
  int NM, MT_gu, MT_d, Rmax, Rh, G, KS_d;
  int dense;  // token-dense gate/up: every tile multiplies all T tokens
  int stages_gu, stages_d;
  size_t smem_gu, smem_d;
};

constexpr size_t kSmemLimit = 227 * 1024;
constexpr size_t kSmemExtra = 1024 /*align*/ + kBarRegion /*barriers & flags*/;

TcGeom tc_geom(const moe_layer_weights& lw, int T, int k) {
  TcGeom g;
  const int TK = T * k;
  const int cap = lw.E < TK ? lw.E : TK;
  const int nmax = T < 256 ? T : 256;
  g.NM = (nmax + 15) & ~15;
  g.MT_gu = (lw.I + kBM - 1) / kBM;
  g.MT_d = (lw.H + kBM - 1) / kBM;
  g.Rmax = TK + 15 * cap;
  // With at most 32 tokens the MMA's N covers every token at once (16 or 32
  // columns, the width a single group would already pad to), so gate/up
  // reads the T token rows directly and the prep kernel needs no union; Hp
  // then holds NM rows per unique expert.
  g.dense = T <= 32 ? 1 : 0;
  g.Rh = g.dense && cap * g.NM > g.Rmax ? cap * g.NM : g.Rmax;
  g.G = sm_count();
  g.KS_d = lw.layout == MOE_LAYOUT_TILED ? 2 : 1;
  const size_t b = static_cast<size_t>(g.NM) * 128;
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

uint32_t pow2_cols(int c) {
  uint32_t v = 32;
  while (v < static_cast<uint32_t>(c)) v <<= 1;
  return v;
}

}  // namespace

bool ffn_tc_supported(const moe_layer_weights& lw, int T, int k) {
  if (lw.dtype != MOE_DTYPE_BF16) return false;
  if (lw.layout != MOE_LAYOUT_ROWMAJOR && lw.layout != MOE_LAYOUT_TILED) return false;
  if (lw.H % kBK || lw.I % kBK) return false;
  if (T < 1 || T > 256) return false;
  TcGeom g = tc_geom(lw, T, k);
  return g.stages_gu >= 2 && g.stages_d >= 2 && encode_fn() != nullptr;
}

size_t ffn_tc_workspace_bytes(const moe_layer_weights& lw, int T, int k) {
  TcGeom g = tc_geom(lw, T, k);
  const int TK = T * k;
  const int cap = lw.E < TK ? lw.E : TK;
  size_t b = 0;
  b += align_up(static_cast<size_t>(g.Rmax) * lw.H * 2, 256);                 // Xp
  b += align_up(static_cast<size_t>(g.Rh) * lw.I * 2, 256);                   // Hp
  b += align_up(static_cast<size_t>(TK) * lw.H * 4, 256);                     // O
  b += align_up(static_cast<size_t>(g.G) * 2 * 2 * g.NM * 128 * 4, 256);       // partials
  b += align_up(static_cast<size_t>(cap + 1) * 4, 256);                       // poff
  b += align_up(static_cast<size_t>(cap) * (g.MT_gu + g.MT_d) * 4, 256);  // fix-up counters
  return b;
}

bool ffn_tc_head_prep(const moe_layer_weights& lw, int T, int k, void* ws, HeadPrep* hp) {
  if (!ffn_tc_supported(lw, T, k) || lw.pool) return false;
  const TcGeom g = tc_geom(lw, T, k);
  if (!g.dense) return false;
  const int TK = T * k;
  const int cap = lw.E < TK ? lw.E : TK;
  char* p = static_cast<char*>(ws);
  hp->xd = reinterpret_cast<uint16_t*>(p);
  p += align_up(static_cast<size_t>(g.Rmax) * lw.H * 2, 256);
  p += align_up(static_cast<size_t>(g.Rh) * lw.I * 2, 256);
  p += align_up(static_cast<size_t>(TK) * lw.H * 4, 256);
  p += align_up(static_cast<size_t>(g.G) * 2 * 2 * g.NM * 128 * 4, 256);
  p += align_up(static_cast<size_t>(cap + 1) * 4, 256);
  hp->counters = reinterpret_cast<int32_t*>(p);
  hp->n_counters = cap * (g.MT_gu + g.MT_d);
  hp->H = lw.H;
  return true;
}

int ffn_tc_launch(const FfnArgs& a) {
  const auto& lw = a.lw;
  const int T = a.T, k = a.k, TK = T * k;
  const int cap = lw.E < TK ? lw.E : TK;
  TcGeom g = tc_geom(lw, T, k);
  char* p = static_cast<char*>(a.ws);
  uint16_t* xp = reinterpret_cast<uint16_t*>(p);
  p += align_up(static_cast<size_t>(g.Rmax) * lw.H * 2, 256);
  uint16_t* hp = reinterpret_cast<uint16_t*>(p);
  p += align_up(static_cast<size_t>(g.Rh) * lw.I * 2, 256);
  float* o = reinterpret_cast<float*>(p);
  p += align_up(static_cast<size_t>(TK) * lw.H * 4, 256);
  float* partials = reinterpret_cast<float*>(p);
  p += align_up(static_cast<size_t>(g.G) * 2 * 2 * g.NM * 128 * 4, 256);
  int32_t* poff = reinterpret_cast<int32_t*>(p);
  p += align_up(static_cast<size_t>(cap + 1) * 4, 256);
  int32_t* cnt_gu = reinterpret_cast<int32_t*>(p);
  int32_t* cnt_d = cnt_gu + static_cast<size_t>(cap) * g.MT_gu;
  const int n_counters = cap * (g.MT_gu + g.MT_d);

  // Tensor maps (host-side encoding only; nothing is enqueued).
  CUtensorMap tm_g, tm_u, tm_x, tm_wd, tm_wd1, tm_h, tm_gt, tm_dt;
  // rows of the last M-tile worth loading (tiled layout): M - 128 (MT - 1), up to a multiple of 8
  auto tail_of = [](uint64_t M) -> int {
    const int r = static_cast<int>(M % kBM);
    return r == 0 ? 0 : ((r + 7) & ~7) < kBM ? ((r + 7) & ~7) : 0;
  };
  const int tail_gu = lw.layout == MOE_LAYOUT_TILED ? tail_of(lw.I) : 0;
  const int tail_d = lw.layout == MOE_LAYOUT_TILED ? tail_of(lw.H) : 0;
  const uint64_t H = lw.H, I = lw.I, E = weight_slots(lw);  // E: expert slots in the buffers
  const uint64_t KBg = H / kBK, KBd = I / kBK;
  if (lw.layout == MOE_LAYOUT_TILED) {
    {
      uint64_t dims[3] = {kBK, 2 * kBM, E * g.MT_gu * KBg}, str[2] = {kBK * 2, 2 * kABytes};
      uint32_t box[3] = {kBK, 2 * kBM, 1};
      if (!make_tmap(&tm_g, lw.w_gate_up, 3, dims, str, box)) return MOE_ERR_CUDA;
      tm_u = tm_g;  // unused: one box carries both gate and up
      tm_gt = tm_g;
      uint32_t boxt[3] = {kBK, static_cast<uint32_t>(tail_gu), 1};
      if (tail_gu && !make_tmap(&tm_gt, lw.w_gate_up, 3, dims, str, boxt)) return MOE_ERR_CUDA;
    }
    {
      uint64_t dims[3] = {kBK, kBM, E * g.MT_d * KBd}, str[2] = {kBK * 2, kABytes};
      uint32_t box2[3] = {kBK, kBM, 2}, box1[3] = {kBK, kBM, 1};
      if (!make_tmap(&tm_wd, lw.w_down, 3, dims, str, box2)) return MOE_ERR_CUDA;
      if (!make_tmap(&tm_wd1, lw.w_down, 3, dims, str, box1)) return MOE_ERR_CUDA;
      tm_dt = tm_wd1;
      uint32_t boxt[3] = {kBK, static_cast<uint32_t>(tail_d), 1};
      if (tail_d && !make_tmap(&tm_dt, lw.w_down, 3, dims, str, boxt)) return MOE_ERR_CUDA;
    }
  } else {
    uint32_t box[3] = {kBK, kBM, 1};
    {
      uint64_t dims[3] = {H, I, E}, str[2] = {H * 2, 2 * I * H * 2};
      if (!make_tmap(&tm_g, lw.w_gate_up, 3, dims, str, box)) return MOE_ERR_CUDA;
      const char* up = static_cast<const char*>(lw.w_gate_up) + I * H * 2;
      if (!make_tmap(&tm_u, up, 3, dims, str, box)) return MOE_ERR_CUDA;
    }
    {
      uint64_t dims[3] = {I, H, E}, str[2] = {I * 2, H * I * 2};
      if (!make_tmap(&tm_wd, lw.w_down, 3, dims, str, box)) return MOE_ERR_CUDA;
      tm_wd1 = tm_wd;
    }
    tm_gt = tm_g;  // unused: rows past the matrix read as zeros without traffic
    tm_dt = tm_wd;
  }
  if (g.dense) {
    // the T token rows; the box's rows past T read as zeros
    uint64_t dims[2] = {H, static_cast<uint64_t>(T)}, str[1] = {H * 2};
    uint32_t box[2] = {kBK, static_cast<uint32_t>(g.NM)};
    if (!make_tmap(&tm_x, xp, 2, dims, str, box)) return MOE_ERR_CUDA;
  } else {
    uint64_t dims[2] = {H, static_cast<uint64_t>(g.Rmax)}, str[1] = {H * 2};
    uint32_t box[2] = {kBK, 16};
    if (!make_tmap(&tm_x, xp, 2, dims, str, box)) return MOE_ERR_CUDA;
  }
  {
    uint64_t dims[2] = {I, static_cast<uint64_t>(g.Rh)}, str[1] = {I * 2};
    uint32_t box[2] = {kBK, 16};
    if (!make_tmap(&tm_h, hp, 2, dims, str, box)) return MOE_ERR_CUDA;
  }

  cudaStream_t s = a.stream;
  if (a.head_prepared) {
    // the layer-head kernel copied the token rows and zeroed the counters
  } else if (g.dense) {
    const long long chunks = static_cast<long long>(T) * (lw.H / 8);
    const long long work = chunks > n_counters ? chunks : n_counters;
    int blocks = static_cast<int>((work + 255) / 256);
    if (blocks > g.G) blocks = g.G;
    LaunchScope ls(kProfPrep, s);
    if (launch_k(ffn_prep_dense_kernel, dim3(blocks), dim3(256), 0, s, a.pdl_first,
                 static_cast<const uint16_t*>(a.x), a.x_rows, a.x_rows_limit, T, lw.H, xp, cnt_gu, n_counters,
                 a.dev_err) != MOE_OK)
      return MOE_ERR_CUDA;
  } else {
    long long chunks = static_cast<long long>(TK) * (lw.H / 8);  // real rows only
    int blocks = static_cast<int>((chunks + 255) / 256);
    if (blocks > g.G * 4) blocks = g.G * 4;
    if (blocks < 1) blocks = 1;
    LaunchScope ls(kProfPrep, s);
    if (launch_k(ffn_prep_kernel, dim3(blocks), dim3(256), 0, s, a.pdl_first,
                 static_cast<const uint16_t*>(a.x), a.x_rows, a.x_rows_limit, T, k, lw.H, cap, a.n_unique,
                 a.offsets, a.perm_token, xp, poff, cnt_gu, n_counters, a.y, a.dev_err) != MOE_OK)
      return MOE_ERR_CUDA;
  }

  TcParams tp{};
  tp.T = T;
  tp.k = k;
  tp.E = lw.E;
  tp.cap = cap;
  tp.NM = g.NM;
  tp.Rmax = g.Rmax;
  tp.Rh = g.Rh;
  tp.dense = g.dense;
  tp.perm_token = a.perm_token;
  tp.ready_flag = a.head_prepared ? a.ready_flag : nullptr;
  tp.ready_value = a.ready_value;
  tp.ready_clear = nullptr;
  tp.n_unique = a.n_unique;
  tp.unique = a.unique;
  tp.offsets = a.offsets;
  tp.poff = poff;
  tp.hp = hp;
  tp.o = o;
  tp.partials = partials;
  tp.dev_err = a.dev_err;
  tp.slot_of = slot_table(lw);
  tp.n_slots = weight_slots(lw);
  tp.tiled = lw.layout == MOE_LAYOUT_TILED ? 1 : 0;
  tp.pdl = 1;
  // Test hook for the failure path (no fault is involved): after
  // moe_test_set_stall(MOE_TEST_STALL_GATE_UP) the gate/up producer issues no
  // copies, every CTA's bounded wait runs out after its budget, and the
  // launch reports MOE_DEV_TIMEOUT with the context intact.
  const bool stall_gu = (test_stall_mask() & MOE_TEST_STALL_GATE_UP) != 0;

  // gate/up
  tp.KS = 1;
  tp.M = lw.I;
  tp.K = lw.H;
  tp.stages = g.stages_gu;
  tp.acc_stages = 2 * 2 * g.NM <= 512 ? 2 : 1;
  tp.tmem_cols = pow2_cols(tp.acc_stages * 2 * g.NM);
  tp.tile_cnt = cnt_gu;
  tp.stall = stall_gu ? 1 : 0;
  if (cudaFuncSetAttribute(ffn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(g.smem_gu)) != cudaSuccess)
    return MOE_ERR_CUDA;
  {
    LaunchScope ls(kProfGateUp, s);
    tp.tail_rows = tail_gu;
    if (launch_k(ffn_tc_kernel<true>, dim3(g.G), dim3(kThreads), g.smem_gu, s, true, tm_g, tm_u, tm_x, tm_gt, tp) !=
        MOE_OK)
      return MOE_ERR_CUDA;
  }

  // down + combine
  tp.pf = a.pf;
  tp.KS = g.KS_d;
  tp.M = lw.H;
  tp.K = lw.I;
  tp.stages = g.stages_d;
  tp.acc_stages = 2 * g.NM <= 512 ? 2 : 1;
  tp.tmem_cols = pow2_cols(tp.acc_stages * g.NM);
  tp.tile_cnt = cnt_d;
  tp.stall = 0;
  tp.ready_clear = tp.ready_flag;
  tp.ready_flag = nullptr;
  if (cudaFuncSetAttribute(ffn_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(g.smem_d)) != cudaSuccess)
    return MOE_ERR_CUDA;
  {
    LaunchScope ls(kProfDown, s);
    tp.tail_rows = tail_d;
    if (launch_k(ffn_tc_kernel<false>, dim3(g.G), dim3(kThreads), g.smem_d, s, true, tm_wd, tm_wd1, tm_h, tm_dt, tp) !=
        MOE_OK)
      return MOE_ERR_CUDA;
  }
  // Weighted combine of the per-(token, slot) outputs, slot order.
  return combine_launch(a, o, true);
}

}  // namespace moe
