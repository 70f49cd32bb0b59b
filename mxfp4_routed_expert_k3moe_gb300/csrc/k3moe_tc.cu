// Expert FFN of the MXFP4 MoE layer on the 5th-generation tensor cores (tcgen05, sm_103a):
//   gate/up:  g = W_gate x, u = W_up x                  (k_tc<GATEUP>)
//             h = SiLU(g) * u and its terms               (the same kernel's epilogue)
//   down:     o_p = w_p W_down h_p                       (k_tc<DOWN>, one row per position p)
//             y[t] = sum_i o_(t,i) + sum_s o_(t,s)        (k_combine)
// The MXFP4 records are consumed as stored (kimi-k3-in-c review, table "KDA·MLA·MoE": the
// experts multiply the 4-bit codes directly): TMA copies 128 rows of a weight matrix into shared
// memory, the E8M0 block scales go to tensor memory, and a block-scaled tcgen05.mma multiplies the
// E2M1 weights (A: M = 128 rows) by the activations (B: N = tokens x terms), applying both scales.
// Two forms, chosen by the token count:
//   - few tokens (fp4): activations as E2M1 terms, kind::mxf4 (K = 64 per MMA); a chunk of the
//     reduction axis is 256 codes = 128 packed bytes per row, copied as is (128-byte swizzle);
//   - more tokens: activations as E4M3 terms, kind::mxf8f6f4 (K = 32 per MMA); a chunk is 128 codes,
//     copied into 16-byte slots of 16 codes (16U4_ALIGN16B). Both chunks take 16 KB per 128 rows.
//
// Activations enter as sums of E4M3 terms: each 32-element block of x (or h) is written as
// v = sum_j q_j 2^{e_j} with q_j E4M3 and 2^{e_j} an E8M0 block scale, each term taking the
// rounding residual of the previous ones. Two terms hold a bf16 block exactly (down to elements
// 2^-13 below the block maximum); three terms leave at most ~2^-12 of the block maximum of an fp32
// x or of h (two terms of h in the bf16-class activation mode). The MMA columns of one token's terms
// are summed in the epilogue.
//
// CTA layout (one CTA per SM, persistent over work items, 384 threads):
//   warps 0-3   epilogue: accumulators (double-buffered in tensor memory) -> per-position sums
//   warps 4-7   loaders: the tensor copy of the weight tile and the bulk copy of its scale words (one
//               lane), the B rows by cp.async, or where a work group's rows are consecutive (the
//               terms of h; the terms of x in position order from 256 tokens) by one more tensor
//               copy, and the B rows' scale words by cp.async; each loader for its own ring slots.
//               On this part one thread issues about one tensor copy per ~500 SM cycles, so a single
//               issuing thread caps the weight stream near 3 TB/s; four reach the DRAM rate.
//   warps 8-11  MMA issuers (one lane each): tcgen05.cp of the scale words into tensor memory, then
//               the MMAs. One issuing thread sustains one tcgen05 instruction per ~120-230 SM cycles
//               whatever N is, so at small N (few tokens) three issuers share the stages, each with
//               its own accumulators in tensor memory; the epilogue adds the partial sums of an item.
// Every ring slot has exactly one agent of each kind (loader v owns the slots s = v mod 4, issuer w
// the slots s = w mod n_iss), so each agent waits on a slot's barriers round after round and a
// parity wait never meets a barrier two phases away.
// The E8M0 scales of the weights are read in the device order (k3moe_pack_records): the scales of a
// stage's chunks of 128 rows are one contiguous block, brought by one bulk copy with the tensor copy
// of the codes. (Fetched row by row, 4 bytes per request, they took a quarter of the DRAM rate.)
// A pipeline stage holds `ch` consecutive 128-code chunks of the reduction axis, brought by one
// tensor copy (the per-copy cost of the TMA unit is amortised over more bytes).
// Each projection has one kernel instance per form; the E2M1 form and the two-term E4M3 rows at
// N = 64 have their tile shapes and ring depths as compile-time constants (the kernels are sensitive
// to every instruction of their per-stage chains), other E4M3 shapes take a general instance.
// Every mbarrier wait is bounded; on a timeout the CTA raises the status word and stops early.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "k3moe_kernels.h"
#include "k3moe_ptx.cuh"

namespace k3 {

namespace {

enum { GATEUP = 0, DOWN = 1 };
constexpr int kMaxIss = 4;                // MMA-issuing warps
constexpr int kLoaders = 4;               // loader warps
constexpr int kWarpLoad = 4, kWarpIss = kWarpLoad + kLoaders, kWarpEnd = kWarpIss + kMaxIss;
constexpr int kThreads = 32 * kWarpEnd;
constexpr int kMaxCh = 2;                 // chunks per stage
constexpr int kTmemCols = 512;
constexpr int kMaxN = 128;               // largest MMA N (B rows per tile)
// TMEM columns per chunk: E4M3 form: A scales at +0..3, B at +16..19 (32 columns); E2M1 form:
// two scale words per row (8 blocks of 32): A at +0..3 and +16..19, B at +32.. and +48.. (64 columns)
constexpr int kMaxStages = 16;
constexpr int kMaxBuf = 4;               // accumulator buffers per issuer
constexpr int kEpRing = 4;               // work groups the epilogue fetches ahead (cp.async)
constexpr int kATile = 128 * 128;        // A tile of a chunk in shared memory (both forms)
constexpr uint32_t kWaitLimit = 1u << 24;  // bound of the drain waits (the pipeline's come with the call)
constexpr uint32_t kPollTestBelow = 64;    // wait bounds below this poll with test_wait (one poll = one test)

using namespace ptx;

// Shared-memory control block (after the pipeline stages).
struct Ctl {
  uint64_t full[kMaxStages];   // weight tiles (TMA bytes), B rows and scale words (cp.async) landed
  uint64_t empty[kMaxStages];  // the stage's MMAs completed
  uint64_t acc_full[kMaxBuf];
  uint64_t acc_empty[kMaxBuf];
  uint64_t drain;
  uint32_t tmem;
  volatile int abort;
  int last;
  alignas(16) WorkGroup ep_wg[4][kEpRing];
  alignas(16) WorkGroup ld_wg[kLoaders][kEpRing];  // loader v's copies of its next items' work groups
  int ld_tok[kLoaders][kEpRing][32];               // ... and the tokens of their positions (gate/up)
  uint32_t ld_row[kLoaders][kMaxN];                // B row n of loader v's current item: activation row, or ~0
};
// Gate/up exchange area after the control block: float [4 epilogue warps][xb_tok tokens][kXb], lane l
// of a warp at [..][..][l]; a row holds 32 values padded to kXb floats, so that a thread reading one
// token's row and its neighbours reading the next tokens' rows fall in distinct banks.
constexpr int kXb = 33;
__host__ __device__ constexpr size_t ctl_bytes() { return (sizeof(Ctl) + 15) / 16 * 16; }

// Position in the ring of pipeline stages: slot s, phase parity of its current round, and whether
// the ring has wrapped at least once.
struct Ring {
  int s = 0;
  uint32_t ph = 0;
  bool wrapped = false;
  __device__ __forceinline__ void next(int S) {
    if (++s == S) {
      s = 0;
      ph ^= 1u;
      wrapped = true;
    }
  }
};

// Bounded wait of the pipeline: at most `limit` polls; on timeout it raises ST_TIMEOUT and the
// CTA-wide abort flag, and every later wait of the CTA returns false at once.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, Ctl* ctl, int* status, uint32_t limit) {
  const bool test = limit < kPollTestBelow;
  for (uint32_t it = 0; it < limit; ++it) {
    if (test ? mbar_test(bar, parity) : mbar_try(bar, parity)) return true;
    if (ctl->abort) return false;
    if (it > 256) __nanosleep(64);
  }
  ctl->abort = 1;
  atomicOr(&status[CTRL_STATUS], ST_TIMEOUT);
  return false;
}

// Wait for copies or MMAs that this CTA started, before it frees the memory they write: bounded by
// kWaitLimit whatever bound the call gave the pipeline, and not cut short by the abort flag.
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t it = 0; it < kWaitLimit; ++it) {
    if (mbar_try(bar, parity)) return true;
    if (it > 256) __nanosleep(64);
  }
  return false;
}

// ------------------------------------------------------------------------------- arguments
// Division by a run-time invariant d through a multiply-high and shifts (the round-up method of
// Granlund and Montgomery, "Division by invariant integers using multiplication", 1994): with
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1, n / d = (t + ((n - t) >> min(l,1))) >> max(l-1,0)
// where t = (m n) >> 32, for every 32-bit n. Item decomposition runs per item in every role, where
// the 64-bit divisions it replaces cost hundreds of cycles.
struct FastDiv {
  uint32_t d, m, s1, s2;
  __host__ void init(uint32_t dv) {
    d = dv;
    uint32_t l = 0;
    while ((1ull << l) < dv) ++l;
    m = (uint32_t)(((1ull << 32) * ((1ull << l) - dv)) / dv + 1);
    s1 = l < 1 ? l : 1;
    s2 = l > 1 ? l - 1 : 0;
  }
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    const uint32_t t = __umulhi(m, n);
    return (t + ((n - t) >> s1)) >> s2;
  }
};

struct TcArgs {
  Cfg c;
  Ws ws;
  const uint8_t* routed;
  const uint8_t* shared;
  float* y;
  long long T;
  int n_tile;   // MMA N (multiple of 16, <= kMaxN)
  int acc_cols; // tensor-memory columns per accumulator (>= n_tile, multiple of 16)
  int n_iss;    // MMA-issuing threads
  int n_acc;    // accumulators per issuer (the MMAs of a chunk alternate between them)
  int n_buf;    // accumulator buffers (items in flight between the issuers and the epilogue)
  int sf_base;  // first column of the scale slots, one per chunk of every stage (after 2 buffers x
                // n_iss x n_acc accumulators)
  int b_bytes;  // shared-memory bytes of the B tile of a chunk
  int ch;       // chunks per stage
  int fp4;      // E2M1 form (kind::mxf4, 256-code chunks) or E4M3 form (kind::mxf8f6f4, 128-code chunks)
  int nch;      // chunks along the reduction axis
  int sf_slot;  // TMEM columns of the scales of a chunk
  int sf_bytes; // shared-memory bytes of the scale words of a chunk
  int terms;    // B rows per token in this kernel (x terms for gate/up, h terms for down)
  int hterms;   // h terms written by the gate/up epilogue
  int xb_tok;   // tokens per item in the gate/up exchange area (0 for the down projection)
  int parts;    // reduction parts per row tile (1: whole items)
  FastDiv div_parts, div_mtiles;
  int stages;   // pipeline depth (<= kMaxStages)
  int tma_b;    // the B rows of a work group, contiguous positions x terms, come by one tensor copy per
                // chunk (map_b: the h terms, or the x terms in position order) instead of cp.async row copies
  int stage_bytes;  // ch x (A tile + B tile + scale words)
};

// Work item: (work group, matrix, 128-row tile, reduction part).
struct Item {
  int wgi, mat, mt, kp, j0, j1;
  WorkGroup wg;
};

// Item geometry only (no work-group read): what the MMA issuers and the epilogue's ring tracking need.
template <int MODE>
__device__ __forceinline__ bool item_geom(const TcArgs& a, long long it, long long n_items, Item& o) {
  if (it >= n_items) return false;
  const int nch = a.nch;
  uint32_t r = (uint32_t)it;
  uint32_t q = a.div_parts.div(r);
  o.kp = (int)(r - q * a.div_parts.d);
  r = q;
  q = a.div_mtiles.div(r);
  o.mt = (int)(r - q * a.div_mtiles.d);
  r = q;
  if (MODE == GATEUP) {
    o.mat = (int)(r & 1u);
    o.wgi = (int)(r >> 1);
  } else {
    o.mat = 0;
    o.wgi = (int)r;
  }
  o.j0 = (int)a.div_parts.div((uint32_t)(o.kp * nch));
  o.j1 = (int)a.div_parts.div((uint32_t)((o.kp + 1) * nch));
  return true;
}

// E8M0 scale bytes of the item's 128-row tile, in the device order (k3moe_pack_records): the tile's
// 128 x K/32 bytes form groups of 512 bytes, one per 4 consecutive blocks; inside a group, the byte
// of row 32c + i and block 4g + e sits at 16 i + 4 c + e. A group is thus the 32 x 16-byte image
// that tcgen05.cp 32x128b.warpx4 spreads to TMEM lane 32q + i, column c: the MMA's scale layout.
template <int MODE>
__device__ __forceinline__ const uint8_t* scale_tile(const TcArgs& a, const Item& it) {
  const Cfg& c = a.c;
  const long long nc = (long long)c.d * c.f / 2, ns = (long long)c.d * c.f / 32;
  const uint8_t* rec = it.wg.expert < c.E ? a.routed + (long long)it.wg.expert * c.stride
                                          : a.shared + (long long)(it.wg.expert - c.E) * c.sstride;
  const int K = MODE == GATEUP ? c.d : c.f;
  const long long off = MODE == GATEUP ? (it.mat == 0 ? nc : 2 * nc + ns) : 2 * (nc + ns) + nc;
  return rec + off + (long long)it.mt * 128 * (K / 32);
}

// B row n of the item (token i = n / terms, term j = n % terms): codes and E8M0 scales.
template <int MODE>
__device__ __forceinline__ bool b_row(const TcArgs& a, const Item& it, int n, const uint8_t*& codes,
                                      const uint8_t*& scales) {
  const Cfg& c = a.c;
  const int i = n / a.terms, j = n - i * a.terms;
  if (i >= it.wg.ntok) return false;
  if (MODE == GATEUP) {
    const long long r = (long long)a.ws.perm_tok[it.wg.pos0 + i] * a.terms + j;
    codes = a.ws.xq + r * c.d;
    scales = a.ws.xs + r * (c.d / 32);
  } else {
    const long long r = (long long)(it.wg.pos0 + i) * a.terms + j;
    codes = a.ws.hq + r * c.f;
    scales = a.ws.hs + r * (c.f / 32);
  }
  return true;
}

// ------------------------------------------------------------------------------- the kernel
// Shared memory of a stage: [A tiles: ch x 16 KB][B tiles: ch x b_bytes][scale words: ch x wpc x 1 KB].
// Scale words: the weight rows' words of every chunk first (word h of chunk cc at 512 (cc wpc + h),
// so that one bulk copy brings them all: they are contiguous in the device order too), then the B
// rows' (word h of chunk cc at 512 (ch wpc + cc wpc + h)). In a 512-byte group the word of row
// 32c + i (4 E8M0 bytes, one per 32-block) sits at byte 16 i + 4 c, the layout that the
// 32x128b.warpx4 copy spreads to TMEM lane 32q + i, column c of every quarter q.
// FORM: the E2M1 form (a.fp4) and the E4M3 form are separate instances, so that each kernel holds only
// its own form's code; the E2M1 form's tile shape, and the E4M3 one of two-term rows with N = 64 (32
// positions or tokens), are compile-time constants in their instances (launch_tc picks and checks).
enum { kFormE4M3 = 0, kFormE2M1 = 1, kFormE4M3N64 = 2 };
template <int MODE, int FORM>
__global__ void __launch_bounds__(kThreads, 1)
    k_tc(const __grid_constant__ CUtensorMap map_r0, const __grid_constant__ CUtensorMap map_r1,
         const __grid_constant__ CUtensorMap map_s0, const __grid_constant__ CUtensorMap map_s1,
         const __grid_constant__ CUtensorMap map_b, TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  // fixed tile shapes: E2M1 six stages of one chunk, three issuers with two accumulator buffers of 16
  // columns, N = 16, 8 terms per activation row; E4M3 N64 four stages of two chunks, two issuers with
  // two buffers of 64 columns, N = 64, 2 terms (the stages: as many as tensor memory holds scale slots)
  constexpr bool F4 = FORM == kFormE2M1, N64 = FORM == kFormE4M3N64;
  const int S = F4 ? 6 : (N64 ? 4 : a.stages), CH = F4 ? 1 : (N64 ? 2 : a.ch);
  const int n_iss = F4 ? 3 : (N64 ? 2 : a.n_iss), n_buf = F4 || N64 ? 2 : a.n_buf, n_acc = F4 || N64 ? 1 : a.n_acc;
  const int acc_cols = F4 ? 16 : (N64 ? 64 : a.acc_cols), n_tile = F4 ? 16 : (N64 ? 64 : a.n_tile);
  const int terms = F4 ? 8 : (N64 ? 2 : a.terms);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + (size_t)S * a.stage_bytes);
  const Cfg& c = a.c;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {  // the maps' descriptors, fetched while the previous kernel finishes
    prefetch_tmap(&map_r0);
    prefetch_tmap(&map_r1);
    prefetch_tmap(&map_s0);
    prefetch_tmap(&map_s1);
    if (!F4 && a.tma_b) prefetch_tmap(&map_b);
  }
  // The gate/up kernel reads the routing, which the previous kernel writes. The down kernel's work
  // groups come from the routing kernel two launches back: it completed before the gate/up kernel
  // (this kernel's predecessor) passed its own grid-dependency wait, hence before this grid was
  // launched. So the down kernel reads its work groups, and its loaders request the weight tiles of
  // the first ring round, before the wait; only the activation rows (h) and everything the epilogue
  // writes come after it.
  if (MODE == GATEUP) pdl_wait();
  pdl_launch_dependents();
  const int n_wg = __ldcg(&a.ws.ctrl[MODE == GATEUP ? CTRL_NWG : CTRL_NWG_DN]);
  const WorkGroup* wgs = MODE == GATEUP ? a.ws.wgs : a.ws.wgs_dn;
  const int nmat = MODE == GATEUP ? 2 : 1;
  const int mtiles = (MODE == GATEUP ? c.f : c.d) / 128;
  const long long n_items = (long long)n_wg * nmat * mtiles * a.parts;
  int* status = a.ws.ctrl;
  const int b_off = CH * kATile, sf_off = CH * (kATile + a.b_bytes);
  const uint32_t tx_chunk = F4 ? 128 * 128 : 128 * 64;  // bytes a chunk's tensor copy delivers
  const int wpc = F4 ? 2 : 1;                            // scale words per row per chunk

  if (n_wg == 0) {  // nothing routed and no shared experts (k_combine writes y = 0)
    if (MODE == DOWN) pdl_wait();
    return;
  }

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&ctl->tmem)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(su32(&ctl->full[s]), 1 + 32);
      mbar_init(su32(&ctl->empty[s]), 1);
    }
    for (int b = 0; b < n_buf; ++b) {
      mbar_init(su32(&ctl->acc_full[b]), n_iss);
      mbar_init(su32(&ctl->acc_empty[b]), 128);
    }
    mbar_init(su32(&ctl->drain), n_iss);
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  const bool loader = warp >= kWarpLoad && warp < kWarpIss;
  if (MODE == DOWN && !loader) pdl_wait();

  if (loader) {
    // ------------------------------------------------------------ loaders (one per slot class)
    // Work groups (kEpRing items ahead) and the tokens of their positions (two items ahead) arrive by
    // cp.async into this loader's ring, so that no load stalls the loader between items (with the
    // DRAM saturated by the weight stream a dependent load waits microseconds).
    const int lv = warp - kWarpLoad;
    const uint64_t pol = policy_evict_first();
    Ring rg;
    bool ok = true;
    WorkGroup* rwg = ctl->ld_wg[lv];
    auto fetch_wg = [&](long long idx, int slot) {  // the work group of item idx, if any
      if (lane == 0 && idx < n_items) {
        Item g;
        item_geom<MODE>(a, idx, n_items, g);
        cp16(su32(&rwg[slot]), &wgs[g.wgi]);
      }
    };
    auto fetch_tok = [&](long long idx, int slot) {  // tokens of item idx's positions (its work group is in `slot`)
      if (MODE == GATEUP && idx < n_items) {
        const WorkGroup g = rwg[slot];
        if (lane < g.ntok && lane < 32) cp4(su32(&ctl->ld_tok[lv][slot][lane]), &a.ws.perm_tok[g.pos0 + lane], 4);
      }
    };
    // Weight codes (tensor copy) and the chunks' A scale groups (one bulk copy each: the groups of a
    // chunk are contiguous in the device order) of chunks j.. of item `it` into stage s, on the
    // stage's full barrier with one arrival.
    auto issue_a = [&](const Item& ia, int j, int s) {
      const bool routed = ia.wg.expert < c.E;
      const CUtensorMap* map = routed ? (ia.mat == 0 ? &map_r0 : &map_r1) : (ia.mat == 0 ? &map_s0 : &map_s1);
      const int ecoord = routed ? ia.wg.expert : ia.wg.expert - c.E;
      const uint8_t* atile = scale_tile<MODE>(a, ia);
      uint8_t* st = smem + (size_t)s * a.stage_bytes;
      mbar_expect_tx(su32(&ctl->full[s]), (tx_chunk + 512 * wpc) * CH);
      tma_load_4d(su32(st), map, 0, ia.mt * 128, j, ecoord, su32(&ctl->full[s]), pol);
      bulk_load(su32(st + sf_off), atile + (size_t)512 * wpc * j, 512 * wpc * CH, su32(&ctl->full[s]), pol);
    };
    // prologue: work groups of the first kEpRing items and tokens of the first two, waited for here
    for (int r = 0; r < kEpRing; ++r) fetch_wg(blockIdx.x + (long long)r * gridDim.x, r);
    asm volatile("cp.async.commit_group;" ::: "memory");
    // Meanwhile the weight tiles of the first ring round (its stages need no empty wait) are requested
    // as soon as their items' work groups are read; the loop below adds their activation rows and
    // scale words. `pre`: global stages of this CTA whose weight tiles are requested here.
    long long pre = 0;
    uint32_t pre_mask = 0;  // this loader's stages among them (bit s)
    if (lane == 0) {
      for (long long ii = blockIdx.x; pre < S && ii < n_items; ii += gridDim.x) {
        Item pi;
        item_geom<MODE>(a, ii, n_items, pi);
        const int4 wv = __ldcg(reinterpret_cast<const int4*>(&wgs[pi.wgi]));
        pi.wg = WorkGroup{wv.x, wv.y, wv.z, wv.w};
        for (int j = pi.j0; j < pi.j1 && pre < S; j += CH, ++pre)
          if ((int)pre % kLoaders == lv) {
            issue_a(pi, j, (int)pre);
            pre_mask |= 1u << pre;
          }
      }
    }
    pre = __shfl_sync(0xffffffffu, pre, 0);
    pre_mask = __shfl_sync(0xffffffffu, pre_mask, 0);
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncwarp();
    if (MODE == DOWN) pdl_wait();
    fetch_tok(blockIdx.x, 0);
    fetch_tok(blockIdx.x + (long long)gridDim.x, 1);
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
    __syncwarp();
    Item it;
    long long kk = 0, gst = 0;  // items, global stages of this CTA
    uint32_t issued = 0;  // bit s: this loader filled slot s at least once; its last round's parity is bit s of `par`
    uint32_t par = 0;
    for (long long ii = blockIdx.x; ok && item_geom<MODE>(a, ii, n_items, it); ii += gridDim.x, ++kk) {
      const int slot = (int)(kk % kEpRing);
      // the group committed two items ago holds this item's tokens and the work group two ahead
      asm volatile("cp.async.wait_group 1;" ::: "memory");
      __syncwarp();
      it.wg = rwg[slot];
      int bsrc[kMaxN / 32];
#pragma unroll
      for (int q = 0; q < kMaxN / 32; ++q) {
        const int n = lane + 32 * q;
        const int i = n / terms;
        bsrc[q] = -1;
        if (n < n_tile && i < it.wg.ntok)
          bsrc[q] = MODE == GATEUP ? ctl->ld_tok[lv][slot][i] : it.wg.pos0 + i;
      }
      __syncwarp();
      // refill: the work group kEpRing ahead into this slot, the tokens of the item two ahead
      fetch_wg(ii + (long long)kEpRing * gridDim.x, slot);
      fetch_tok(ii + 2LL * gridDim.x, (int)((kk + 2) % kEpRing));
      asm volatile("cp.async.commit_group;" ::: "memory");
      // B row n of the tile = activation row (token or position) * terms + term; the rows' indices go
      // to this loader's table, which the code copies below read, and the scale pointers of rows
      // lane + 32 q stay in registers
      const int kk = MODE == GATEUP ? c.d : c.f;
      const long long row_bytes = F4 ? kk / 2 : kk;
      const uint8_t* bbase = MODE == GATEUP ? a.ws.xq : a.ws.hq;
      uint32_t* rtab = ctl->ld_row[lv];
      const int nrows = min(n_tile, it.wg.ntok * terms);  // rows past these are not read
      const uint8_t* bscales[kMaxN / 32];
#pragma unroll
      for (int q = 0; q < kMaxN / 32; ++q) {
        bscales[q] = nullptr;
        const int n = lane + 32 * q;
        uint32_t r = ~0u;  // (rows < 3 * 2^30: positions < 2^30, at most 3 terms above 2 tokens)
        if (bsrc[q] >= 0) {
          r = (uint32_t)bsrc[q] * (uint32_t)terms + (uint32_t)(n - (n / terms) * terms);
          bscales[q] = (MODE == GATEUP ? a.ws.xs : a.ws.hs) + (long long)r * (kk / 32);
        }
        if (n < n_tile) rtab[n] = r;
      }
      __syncwarp();
      for (int j = it.j0; j < it.j1; j += CH, rg.next(S)) {
        const int s = rg.s;
        const long long g = gst++;
        if (s % kLoaders != lv) continue;
        if (rg.wrapped)
          ok = __all_sync(0xffffffffu, wait_bar(su32(&ctl->empty[s]), rg.ph ^ 1u, ctl, status, c.wait_limit));
        if (!ok) break;
        issued |= 1u << s;
        par = (par & ~(1u << s)) | (rg.ph << s);
        uint8_t* st = smem + (size_t)s * a.stage_bytes;
        if (lane == 0) {
          if (g >= pre) issue_a(it, j, s);
          if (!F4 && a.tma_b) {  // the work group's B rows of the stage's chunks: n_tile rows from position pos0 on
            mbar_expect_tx_only(su32(&ctl->full[s]), (uint32_t)(n_tile * 128 * CH));
            tma_load_3d(su32(st + b_off), &map_b, 0, it.wg.pos0 * terms, j, su32(&ctl->full[s]));
          }
        }
        for (int cc = 0; cc < CH; ++cc) {
          const int jj = j + cc;
          const uint32_t sb = su32(st + b_off + cc * a.b_bytes);
          const uint32_t sc = su32(st + sf_off) + 512 * wpc * (CH + cc);  // B rows' scale words of the chunk
          // codes: lane = 16-byte segment k16 of row 4 it + lane / 8, so that one copy instruction
          // reads four 128-byte rows (one row per lane read 32 rows: a quarter of the L1 rate)
          // (four rows per lane at a time: their table reads are issued before the copies)
          const int k16 = lane & 7;
          for (int n0 = lane >> 3; n0 < nrows && !(!F4 && a.tma_b); n0 += 16) {
            uint32_t r[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) r[u] = n0 + 4 * u < nrows ? rtab[n0 + 4 * u] : ~0u;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int n = n0 + 4 * u;
              if (r[u] != ~0u)
                cp16(sb + n * 128 + ((k16 ^ (n & 7)) << 4), bbase + (long long)r[u] * row_bytes + jj * 128 + k16 * 16);
            }
          }
#pragma unroll
          for (int q = 0; q < kMaxN / 32; ++q)
            if (bscales[q])
              for (int h = 0; h < wpc; ++h)
                cp4(sc + 512 * h + 16 * lane + 4 * q, bscales[q] + 4 * (wpc * jj + h), 4);
        }
        cp_arrive_noinc(su32(&ctl->full[s]));
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    // after a timeout: the last fill of each of this loader's slots (tensor and bulk copies, and the
    // lanes' cp.async, all counted by the slot's full barrier) lands before the CTA frees its memory.
    // Earlier fills of a slot have landed: the slot was refilled only after their MMAs completed. A
    // slot of the first round whose weight tiles were requested early but which the loop did not
    // reach gets the lanes' arrivals here, so that its barrier completes when those tiles land.
    if (!ok) {
      const uint32_t unreached = pre_mask & ~issued;
      for (int s = 0; s < S; ++s)
        if ((unreached >> s) & 1u) cp_arrive_noinc(su32(&ctl->full[s]));
      if (lane == 0)
        for (int s = 0; s < S; ++s)
          if (((issued | unreached) >> s) & 1u) drain_wait(su32(&ctl->full[s]), ((par & issued) >> s) & 1u);
    }
    __syncwarp();
  } else if (warp >= kWarpIss) {
    // ------------------------------------------------------------ MMA issuers
    const int w = warp - kWarpIss;
    if (lane == 0 && w < n_iss) {
      // instruction descriptor: A/B formats (mxf4: E2M1 = 1; mxf8f6f4: A E2M1 = 5, B E4M3 = 0), N, UE8M0, M
      const uint32_t idesc = (F4 ? ((1u << 7) | (1u << 10)) : (5u << 7)) | ((uint32_t)(n_tile >> 3) << 17) |
                             (1u << 23) | ((uint32_t)(128 >> 4) << 24);
      // descriptors of stage 0, chunk 0; stage s / chunk cc add their byte offsets / 16 to the
      // start-address field
      const uint64_t da0 = sw128_desc(su32(smem)), db0 = sw128_desc(su32(smem) + b_off);
      const uint64_t dsa0 = sf_desc(su32(smem) + sf_off);
      const int wpc = F4 ? 2 : 1;
      const uint32_t st16 = (uint32_t)a.stage_bytes >> 4, bb16 = (uint32_t)a.b_bytes >> 4;
      long long i = 0;
      Ring rg;
      Item it;
      bool ok = true;
      for (long long ii = blockIdx.x; ok && item_geom<MODE>(a, ii, n_items, it); ii += gridDim.x, ++i) {
        const long long rb = i / n_buf;  // the buffer's round
        const int b = (int)(i - rb * n_buf);
        if (rb > 0 && !wait_bar(su32(&ctl->acc_empty[b]), (uint32_t)((rb - 1) & 1), ctl, status, c.wait_limit)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)((b * n_iss + w) * n_acc * acc_cols);
        uint32_t started = 0;  // bit h: accumulator h already holds a partial sum of this item
        for (int j = it.j0; j < it.j1; j += CH, rg.next(S)) {
          const int s = rg.s;
          if (s % n_iss != w) continue;
          if (!wait_bar(su32(&ctl->full[s]), rg.ph, ctl, status, c.wait_limit)) { ok = false; break; }
          tc_fence_after();
          fence_async_smem();  // B rows and scale words arrived through cp.async (generic proxy)
          const uint64_t so = (uint64_t)(s * st16);
          for (int cc = 0; cc < CH; ++cc) {
            // scale words of the chunk: A word w to column col + 16 w, B word w to col + 16 (wpc + w)
            // The scale slot belongs to the stage: it is rewritten only after the stage's previous MMAs
            // completed (the loader refilled the stage after its empty barrier).
            const uint32_t col = tmem + (uint32_t)(a.sf_base + (s * CH + cc) * a.sf_slot);
            for (int w2 = 0; w2 < 2 * wpc; ++w2) {
              const int grp = w2 < wpc ? cc * wpc + w2 : (CH + cc) * wpc + (w2 - wpc);  // 512-byte group
              tc_cp_32x128b_x4(col + 16 * w2, dsa0 + so + (uint64_t)(grp * (512 >> 4)));
            }
            const uint64_t da = da0 + so + (uint64_t)(cc * (kATile >> 4)), db = db0 + so + (uint64_t)(cc * bb16);
            if (F4) {
              // K = 64 per MMA; MMA k uses scale word k / 2, byte pair 2 (k % 2)
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint32_t hw = (uint32_t)(k >> 1), sf = (uint32_t)(k & 1) * 2u;
                tc_mma_f4(d, da + 2 * k, db + 2 * k, idesc | (sf << 4) | (sf << 29), col + 16 * hw, col + 32 + 16 * hw,
                          started & 1u);
                started = 1;
              }
            } else {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int h = k & (n_acc - 1);
                tc_mma(d + (uint32_t)(h * acc_cols), da + 2 * k, db + 2 * k,
                       idesc | ((uint32_t)k << 4) | ((uint32_t)k << 29), col, col + 16, (started >> h) & 1u);
                started |= 1u << h;
              }
            }
          }
          tc_commit(su32(&ctl->empty[s]));
        }
        if (!ok) break;
        tc_commit(su32(&ctl->acc_full[b]));
      }
      tc_commit(su32(&ctl->drain));  // every MMA issued above has completed when this arrives
      drain_wait(su32(&ctl->drain), 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 0-3)
    // Per item: the partial accumulators of a 16-column block are read with one wait, the buffer is
    // released right after the last block is read, and only then are the sums formed and stored. The
    // work group of the item two ahead (and the gate weights of the next one) are read while the
    // current one is waited for: while the weight stream saturates the DRAM, a read that misses L2
    // waits microseconds.
    const int q = warp;
    float* xb = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ctl) + ctl_bytes());  // gate/up exchange
    long long i = 0;
    int bad = 0;
    int g0 = 0;  // ring slot of the item's first stage
    Item it;
    // the work groups of the next kEpRing items arrive by cp.async into this warp's ring, so that
    // no load sits in the epilogue's path (with the DRAM saturated a plain load waited ~2 us)
    auto fetch_wg = [&](long long idx, int slot) {
      if (lane == 0 && idx < n_items) {
        Item g;
        item_geom<MODE>(a, idx, n_items, g);
        cp16(su32(&ctl->ep_wg[q][slot]), &wgs[g.wgi]);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    for (int r = 0; r < kEpRing; ++r) fetch_wg(blockIdx.x + (long long)r * gridDim.x, r);
    for (long long ii = blockIdx.x; item_geom<MODE>(a, ii, n_items, it); ii += gridDim.x, ++i) {
      const int slot = (int)(i % kEpRing);
      asm volatile("cp.async.wait_group %0;" ::"n"(kEpRing - 1) : "memory");
      __syncwarp();
      it.wg = ctl->ep_wg[q][slot];
      __syncwarp();
      fetch_wg(ii + (long long)kEpRing * gridDim.x, slot);  // reuses the slot just read
      const int nst = (it.j1 - it.j0) / CH;  // stages of the item
      const long long rb = i / n_buf;
      const int b = (int)(i - rb * n_buf);
      bool okw =
          __all_sync(0xffffffffu, wait_bar(su32(&ctl->acc_full[b]), (uint32_t)(rb & 1), ctl, status, c.wait_limit));
      // gate/up: the four warps agree (they meet at a barrier below); this also keeps the exchange
      // area of the previous item until every warp has read it
      if (MODE == GATEUP) okw = bar_and(1, 128, okw);
      if (!okw) break;
      tc_fence_after();
      const int row = it.mt * 128 + 32 * q + lane;
      const int ncols = it.wg.ntok * terms;
      // issuers that received stages: owners (slot mod n_iss) of slots g0, g0 + 1, ...; their partial
      // sums are added in issuer order
      unsigned mask = 0;
      for (int t = 0, sl = g0; t < nst && t < S; ++t, sl = (sl + 1 == S) ? 0 : sl + 1) mask |= 1u << (sl % n_iss);
      const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * n_iss * acc_cols);
      float run = 0.0f;
      bool nan_row = false;
      int tk = 0, jt = 0;  // token and term of the current column
      // at the smallest N (four issuers of 16 columns, one token's terms) one load takes all partials:
      // every tensor-memory load waits in the tensor pipe with the MMAs, so fewer loads cost less
      const bool one_load = n_iss * acc_cols == 64 && ncols <= 16;
      for (int cb = 0; cb < ncols; cb += 16) {
        uint32_t u[kMaxIss][16];
        if (one_load) {
          tc_ld64(lane_base, &u[0][0]);
        } else {
#pragma unroll
          for (int w = 0; w < kMaxIss; ++w)
            if ((mask >> w) & 1u) tc_ld16(lane_base + (uint32_t)(w * acc_cols + cb), u[w]);
        }
        tc_wait_ld();
        if (cb + 16 >= ncols) {  // buffer read completely: hand it back
          tc_fence_before();
          mbar_arrive(su32(&ctl->acc_empty[b]));
        }
        float v[16];
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) v[cc] = 0.0f;
#pragma unroll
        for (int w = 0; w < kMaxIss; ++w)
          if ((mask >> w) & 1u) {
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) v[cc] += __uint_as_float(u[w][cc]);
          }
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
          const int col = cb + cc;
          if (col < ncols) {
            run += v[cc];
            if (++jt == terms) {
              jt = 0;
              const long long pos = it.wg.pos0 + tk;
              nan_row |= (run != run);
              if (MODE == GATEUP)
                xb[(q * a.xb_tok + tk) * kXb + lane] = run;
              else
                a.ws.part[pos * c.d + row] = run;  // the gate weight is applied by the combine
              run = 0.0f;
              ++tk;
            }
          }
        }
      }
      // activations are finite by construction, so a NaN sum means a NaN weight scale: find it
      if (nan_row) {
        const uint8_t* sg = scale_tile<MODE>(a, it) + 16 * lane + 4 * q;  // row 32 q + lane of the tile
        for (int g = it.j0 * wpc; g < it.j1 * wpc; ++g)
          bad |= (__vcmpeq4(__ldg(reinterpret_cast<const unsigned*>(sg + (size_t)512 * g)), 0xFFFFFFFFu) != 0u);
      }
      if (MODE == GATEUP) {
        // The stacked tile's rows 0-63 are gate rows and 64-127 the up rows of the same 64 rows of h
        // (k3moe_pack_records): warp q and warp q ^ 2 hold g and u of h rows 32 (q & 1) + lane of
        // them. After the exchange, warps 0-1 finish the even tokens of the item, warps 2-3 the odd.
        bar_sync(1, 128);
        const int p = q & 1;
        const int nb = c.f / 32, blk = 4 * it.mt + 2 * it.mat + p;  // 32-block of h
        if (F4) {
          for (int i = q >> 1; i < it.wg.ntok; i += 2) {
            const float g = xb[(p * a.xb_tok + i) * kXb + lane], u = xb[((p + 2) * a.xb_tok + i) * kXb + lane];
            const long long pos = it.wg.pos0 + i;
            split_terms_fp4(silu(g) * u, c.hterms, a.ws.hq + (pos * c.hterms) * (c.f / 2) + blk * 16, c.f / 2,
                            a.ws.hs + (pos * c.hterms) * nb + blk, nb, lane);
          }
        } else {
          // E4M3 terms: one thread per (token, 32-row half of h): its block's 32 values of g and u, h,
          // and the terms of the block in registers, the steps of split_terms element by element (the
          // block maximum as a loop, not as a chain of warp shuffles per term and token)
          const int t = 32 * q + lane;
          if (t < 2 * it.wg.ntok) {
            const int i = t >> 1, hp = t & 1;
            const float* gs = xb + (hp * a.xb_tok + i) * kXb;
            const float* us = xb + ((hp + 2) * a.xb_tok + i) * kXb;
            float r[32];
            float amax = 0.0f;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              r[e] = silu(gs[e]) * us[e];
              amax = fmaxf(amax, fabsf(r[e]));
            }
            const int hblk = 4 * it.mt + 2 * it.mat + hp;
            const long long pos = it.wg.pos0 + i;
            uint8_t* cdst = a.ws.hq + (pos * c.hterms) * c.f + hblk * 32;
            uint8_t* sdst = a.ws.hs + (pos * c.hterms) * nb + hblk;
            for (int j = 0; j < c.hterms; ++j) {
              int e = 0;
              if (amax > 0.0f && amax <= 3.402823466e38f) e = ilogbf(amax) - 7;
              e = e < -127 ? -127 : (e > 127 ? 127 : e);
              const float sc = pow2i(-e), back = pow2i(e);
              uint32_t w[8];
              float nmax = 0.0f;
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                uint16_t q2;
                asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(q2) : "f"(r[2 * k + 1] * sc), "f"(r[2 * k] * sc));
                uint32_t h2;
                asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(q2));
                r[2 * k] -= __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))) * back;
                r[2 * k + 1] -= __half2float(__ushort_as_half((unsigned short)(h2 >> 16))) * back;
                nmax = fmaxf(nmax, fmaxf(fabsf(r[2 * k]), fabsf(r[2 * k + 1])));
                if (k & 1) w[k >> 1] |= (uint32_t)q2 << 16;
                else w[k >> 1] = q2;
              }
              uint4* cv = reinterpret_cast<uint4*>(cdst + (long long)j * c.f);
              cv[0] = make_uint4(w[0], w[1], w[2], w[3]);
              cv[1] = make_uint4(w[4], w[5], w[6], w[7]);
              sdst[(long long)j * nb] = (uint8_t)(e + 127);
              amax = nmax;
            }
          }
        }
      }
      g0 = (g0 + nst) % S;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (bad) atomicOr(&status[CTRL_STATUS], ST_NAN_SCALE);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

// ------------------------------------------------------------------------------- combine
// y[t] = sum over the top-k slots of t (in slot order) of the gate-weighted expert outputs, then the
// shared experts; one thread per (token, row of d_model). BATCH (few tokens, where the kernel is one
// chain of dependent loads): a thread issues all its loads before the sums, in two rounds (the slots'
// positions, then their gate weights and outputs), and adds in the same order; measured 0.9 us
// faster per layer at one token, but its registers halve the occupancy, which made it slower from
// 64 tokens on (4096 tokens: 0.33 ms).
constexpr int kCombMaxK = 32, kCombMaxS = 8;  // top_k <= 32, n_shared <= 8 (checked by the API)
// SB: the shared experts are bf16 ones, whose outputs come as partial sums in ws.sho (its own instance,
// so that the MXFP4 path keeps its registers and occupancy).
constexpr long long kCombBatchMaxT = 2;
template <bool BATCH, bool SB>
__global__ void __launch_bounds__(256) k_combine(Cfg c, Ws ws, float* y, long long T) {
  pdl_wait();
  pdl_launch_dependents();
  const long long P_R = T * c.k;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < T * c.d;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long tok = idx / c.d;
    const int row = (int)(idx - tok * c.d);
    if (!BATCH) {
      float s = 0.0f;
      for (int i = 0; i < c.k; ++i) {
        const int p = ws.inv[tok * c.k + i];
        if (p >= 0) s += ws.perm_w[p] * ws.part[(long long)p * c.d + row];
      }
      for (int sh = 0; sh < c.S; ++sh) s += ws.part[(P_R + (long long)sh * T + tok) * c.d + row];
      if (SB)
        for (int sb = 0; sb < c.Sb; ++sb)
          for (int z = 0; z < c.nsp2; ++z) s += ws.sho[((long long)(sb * c.nsp2 + z) * T + tok) * c.d + row];
      y[idx] = s;
      continue;
    }
    int p[kCombMaxK];
#pragma unroll
    for (int i = 0; i < kCombMaxK; ++i) p[i] = i < c.k ? __ldcg(&ws.inv[tok * c.k + i]) : -1;
    float w[kCombMaxK], o[kCombMaxK], so[kCombMaxS];
#pragma unroll
    for (int i = 0; i < kCombMaxK; ++i) {
      w[i] = 0.0f;
      o[i] = 0.0f;
      if (p[i] >= 0) {
        w[i] = __ldcg(&ws.perm_w[p[i]]);
        o[i] = __ldcg(&ws.part[(long long)p[i] * c.d + row]);
      }
    }
#pragma unroll
    for (int sh = 0; sh < kCombMaxS; ++sh)
      so[sh] = sh < c.S ? __ldcg(&ws.part[(P_R + (long long)sh * T + tok) * c.d + row]) : 0.0f;
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kCombMaxK; ++i)
      if (p[i] >= 0) s += w[i] * o[i];
#pragma unroll
    for (int sh = 0; sh < kCombMaxS; ++sh)
      if (sh < c.S) s += so[sh];
    if (SB)
      for (int sb = 0; sb < c.Sb; ++sb)
        for (int z = 0; z < c.nsp2; ++z) s += __ldcg(&ws.sho[((long long)(sb * c.nsp2 + z) * T + tok) * c.d + row]);
    y[idx] = s;
  }
}

// ------------------------------------------------------------------------------- device order
// Byte of row r (of 128) and 32-block b inside the scale image of one 128-row tile (k3moe.h): the
// 512-byte group of blocks 4g..4g+3 holds, at 16 i + 4 c + e, row 32 c + i and block 4 g + e.
__device__ __forceinline__ int img_at(int r, int b) { return 512 * (b >> 2) + 16 * (r & 31) + 4 * (r >> 5) + (b & 3); }

// Converts whole records between the stored order and the device order read by k_tc. One CTA per
// unit, in place:
//   gate/up pair u (gate rows 128u..128u+127 and up rows 128u..128u+127): the codes of gate rows
//     128u+64.. and up rows 128u.. swap places (64 rows each; the swap is its own inverse), and the
//     scale bytes of both tiles, staged in shared memory, are written as the images of the stacked
//     tiles 2u (gate rows 128u.., then up rows 128u..) and 2u+1 (gate rows 128u+64.., up rows
//     128u+64..) into the ranges of gate tile u and up tile u (or back);
//   down tile t: its scale bytes are written as the tile's image (or back).
__global__ void __launch_bounds__(256) k_pack_records(uint8_t* records, long long n_rec, long long stride, int d,
                                                       int f, int to_device) {
  extern __shared__ __align__(16) uint8_t sbuf[];
  const int pairs = f / 128, tiles_dn = d / 128;
  const long long per_rec = (long long)pairs + tiles_dn;
  const long long nc = (long long)d * f / 2, ns = (long long)d * f / 32;
  for (long long unit = blockIdx.x; unit < n_rec * per_rec; unit += gridDim.x) {
    const long long rr = unit / per_rec;
    const int t = (int)(unit - rr * per_rec);
    uint8_t* rec = records + rr * stride;
    if (t < pairs) {
      const int nb = d / 32;  // blocks per row, a multiple of 4
      const int n = 128 * nb;
      uint8_t* gs = rec + nc + (long long)t * n;            // gate tile t's scale range
      uint8_t* us = rec + 2 * nc + ns + (long long)t * n;   // up tile t's scale range
      uint8_t* gc = rec + ((long long)t * 128 + 64) * (d / 2);     // gate rows 128t+64.. (codes)
      uint8_t* uc = rec + nc + ns + (long long)t * 128 * (d / 2);  // up rows 128t..
      for (int o = threadIdx.x * 16; o < 64 * (d / 2); o += blockDim.x * 16) {
        const uint4 x = *reinterpret_cast<const uint4*>(gc + o), y = *reinterpret_cast<const uint4*>(uc + o);
        *reinterpret_cast<uint4*>(gc + o) = y;
        *reinterpret_cast<uint4*>(uc + o) = x;
      }
      for (int o = threadIdx.x * 16; o < n; o += blockDim.x * 16) {
        *reinterpret_cast<uint4*>(sbuf + o) = *reinterpret_cast<const uint4*>(gs + o);
        *reinterpret_cast<uint4*>(sbuf + n + o) = *reinterpret_cast<const uint4*>(us + o);
      }
      __syncthreads();
      for (int o = threadIdx.x; o < 2 * n; o += blockDim.x) {
        const int h = o >= n, oo = o - h * n;  // destination: gate range (h 0) or up range (h 1)
        int src;
        if (to_device) {  // oo is byte img_at(r, b) of stacked tile 2t + h
          const int g = oo >> 9, i = (oo >> 4) & 31, c = (oo >> 2) & 3, e = oo & 3;
          const int r = 32 * c + i, b = 4 * g + e;
          const int row = 64 * h + (r & 63);   // row of the gate (r < 64) or up tile
          src = (r < 64 ? 0 : n) + row * nb + b;
        } else {  // oo = row * nb + b of the gate (h 0) or up (h 1) tile t
          const int row = oo / nb, b = oo - row * nb;
          const int st = row >> 6;             // stacked tile 2t + st holds the row ...
          const int r = 64 * h + (row & 63);   // ... as its row r
          src = st * n + img_at(r, b);
        }
        (h ? us : gs)[oo] = sbuf[src];
      }
      __syncthreads();
    } else {
      const int nb = f / 32;
      const int n = 128 * nb;
      uint8_t* base = rec + 2 * (nc + ns) + nc + (long long)(t - pairs) * n;
      for (int o = threadIdx.x * 16; o < n; o += blockDim.x * 16)
        *reinterpret_cast<uint4*>(sbuf + o) = *reinterpret_cast<const uint4*>(base + o);
      __syncthreads();
      for (int o = threadIdx.x; o < n; o += blockDim.x) {
        int src;
        if (to_device) {
          const int g = o >> 9, i = (o >> 4) & 31, c = (o >> 2) & 3, e = o & 3;
          src = (32 * c + i) * nb + 4 * g + e;
        } else {
          const int row = o / nb, b = o - row * nb;
          src = img_at(row, b);
        }
        base[o] = sbuf[src];
      }
      __syncthreads();
    }
  }
}

// ------------------------------------------------------------------------------- host side
int g_sms = 0;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_mu;

cudaError_t get_encode() {
  if (g_encode) return cudaSuccess;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return e != cudaSuccess ? e : cudaErrorNotSupported;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return cudaSuccess;
}

// 3D map over expert records: {K codes, rows, experts}, 128 x 128 boxes of 16U4_ALIGN16B codes.
struct MapKey {
  const void* base;
  long long K, rows, experts, stride;
  int ch, fp4;
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool used;
};
constexpr int kMapCache = 64;
MapEntry g_maps[kMapCache];
int g_map_next = 0;

// 4D map over one weight matrix of every expert record, boxes of 128 rows x `ch` chunks landing as
// ch tiles of 16 KB with the 128-byte swizzle:
//   E4M3 form: {128 codes of a chunk, rows, K/128 chunks, experts}, strides {K/2, 64, record} bytes,
//              16U4_ALIGN16B (16 codes per 16-byte slot);
//   E2M1 form: {128 bytes (256 codes) of a chunk, rows, K/256 chunks, experts}, strides {K/2, 128,
//              record}, bytes as stored.
cudaError_t weight_map(const uint8_t* base, long long K, long long rows, long long experts, long long stride, int ch,
                       int fp4, CUtensorMap* out) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (auto& m : g_maps)
    if (m.used && m.key.base == base && m.key.K == K && m.key.rows == rows && m.key.experts == experts &&
        m.key.stride == stride && m.key.ch == ch && m.key.fp4 == fp4) {
      *out = m.map;
      return cudaSuccess;
    }
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  MapEntry& m = g_maps[g_map_next];
  g_map_next = (g_map_next + 1) % kMapCache;
  cuuint64_t gdim[4] = {128, (cuuint64_t)rows, (cuuint64_t)(K / (fp4 ? 256 : 128)), (cuuint64_t)(experts > 0 ? experts : 1)};
  cuuint64_t gstride[3] = {(cuuint64_t)(K / 2), (cuuint64_t)(fp4 ? 128 : 64), (cuuint64_t)stride};
  cuuint32_t box[4] = {128, 128, (cuuint32_t)ch, 1}, estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(&m.map, fp4 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4,
                        const_cast<uint8_t*>(base), gdim, gstride,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    m.used = false;
    return cudaErrorInvalidValue;
  }
  m.key = MapKey{base, K, rows, experts, stride, ch, fp4};
  m.used = true;
  *out = m.map;
  return cudaSuccess;
}

// Bytes of the gate/up exchange area (float per epilogue warp, token and lane).
size_t xb_bytes(const TcArgs& a) { return ((size_t)4 * a.xb_tok * kXb * sizeof(float) + 15) / 16 * 16; }

template <int MODE>
cudaError_t launch_tc(const TcArgs& a, const CUtensorMap& r0, const CUtensorMap& r1, const CUtensorMap& s0,
                      const CUtensorMap& s1, const CUtensorMap& b, long long items_max, cudaStream_t st) {
  if (items_max >= (1LL << 31)) return cudaErrorInvalidValue;  // item indices are decomposed in 32 bits
  // the E2M1 instance compiles its tile shape in; so does the E4M3 N64 one, taken when the shape is its
  const bool n64 = !a.fp4 && a.stages == 4 && a.ch == 2 && a.n_iss == 2 && a.n_buf == 2 && a.n_acc == 1 &&
                   a.acc_cols == 64 && a.n_tile == 64 && a.terms == 2;
  if (a.fp4 && (a.stages != 6 || a.ch != 1 || a.n_iss != 3 || a.n_buf != 2 || a.n_acc != 1 || a.acc_cols != 16 ||
                a.n_tile != 16 || a.terms != 8))
    return cudaErrorInvalidConfiguration;
  const size_t smem = (size_t)a.stages * a.stage_bytes + ctl_bytes() + xb_bytes(a) + 1024;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_tc<MODE, kFormE2M1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_tc<MODE, kFormE4M3>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_tc<MODE, kFormE4M3N64>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  long long grid = items_max < g_sms ? items_max : g_sms;
  if (grid < 1) grid = 1;
  return launch_pdl(a.fp4 ? k_tc<MODE, kFormE2M1> : (n64 ? k_tc<MODE, kFormE4M3N64> : k_tc<MODE, kFormE4M3>),
                    dim3((unsigned)grid), dim3(kThreads), smem, st, r0, r1, s0, s1, b, a);
}

// Tile geometry for an MMA N of n_tile: TMEM holds two accumulator buffers per issuer and then one
// scale slot per chunk of every stage, which bounds the ring's depth; shared memory holds the stages
// and the control block. (Scale slots owned by the issuers instead, with a deeper ring in shared
// memory, measured slower: an issuer then waits for its own earlier MMAs.)
// Chunks per stage: kMaxCh when every item's chunk range divides evenly, else 1.
int chunks_per_stage(long long nch, long long parts) {
  return (nch % parts == 0 && (nch / parts) % kMaxCh == 0) ? kMaxCh : 1;
}

// With fewer than 4 stages of ch chunks the stage shrinks to one chunk.
void size_tiles(TcArgs& a, int ch, int mtiles) {
  a.sf_slot = a.fp4 ? 64 : 32;
  a.sf_bytes = a.fp4 ? 2048 : 1024;
  a.div_parts.init((uint32_t)a.parts);
  a.div_mtiles.init((uint32_t)mtiles);
  a.acc_cols = 16;  // a power of two >= n_tile: every accumulator starts at a multiple of its width
  while (a.acc_cols < a.n_tile) a.acc_cols *= 2;
  // issuers and accumulator buffers: small N needs several issuers (issue rate); three (each owning
  // two of the six stages at N = 16) measured faster than four (two owning two, two owning one) or
  // two. Above 64 columns: with few tokens per work group (T < 256) two issuers with one buffer each
  // (measured faster), at prefill sizes one issuer with two buffers (deeper ring, overlapped epilogue)
  a.n_iss = a.n_tile <= 32 ? 3 : (a.n_tile <= 64 || a.T < 256 ? 2 : 1);
  a.n_acc = 1;  // two alternating accumulators measured no faster at any N
  a.n_buf = (a.n_tile <= 64 || a.T >= 256) ? 2 : 1;  // (three, with a stage fewer, measured no faster)
  a.sf_base = (a.n_buf * a.n_iss * a.n_acc * a.acc_cols + 31) / 32 * 32;
  a.b_bytes = (a.n_tile * 128 + 1023) / 1024 * 1024;
  for (;; ch = 1) {
    a.ch = ch;
    a.stage_bytes = ch * (kATile + a.b_bytes + a.sf_bytes);
    int st = (227 * 1024 - 1024 - (int)ctl_bytes() - (int)xb_bytes(a)) / a.stage_bytes;
    const int tm = (kTmemCols - a.sf_base) / (a.sf_slot * ch);
    if (st > tm) st = tm;
    if (st > kMaxStages) st = kMaxStages;
    a.stages = st;
    if (st >= 4 || ch == 1) break;
  }
}

int round16(int v) { return (v + 15) / 16 * 16; }

}  // namespace

namespace {

struct TcMaps {
  CUtensorMap gr, ur, gs, us, dr, ds;
};

cudaError_t setup(const Cfg& c, const uint8_t* routed, const uint8_t* shared, int ch_gu, int ch_dn, TcMaps& m,
                  const uint8_t*& sh) {
  const int f4 = c.fp4;
  if (g_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_sms <= 0) g_sms = 1;
  }
  const long long nc = (long long)c.d * c.f / 2, ns = (long long)c.d * c.f / 32;
  sh = (c.S > 0 && shared) ? shared : routed;
  const long long sh_n = c.S > 0 ? c.S : 1;
  const long long sh_stride = (c.S > 0 && shared) ? c.sstride : c.stride;
  cudaError_t e;
  if (ch_gu > 0) {
    if ((e = weight_map(routed, c.d, c.f, c.E, c.stride, ch_gu, f4, &m.gr)) != cudaSuccess) return e;
    if ((e = weight_map(routed + nc + ns, c.d, c.f, c.E, c.stride, ch_gu, f4, &m.ur)) != cudaSuccess) return e;
    if ((e = weight_map(sh, c.d, c.f, sh_n, sh_stride, ch_gu, f4, &m.gs)) != cudaSuccess) return e;
    if ((e = weight_map(sh + nc + ns, c.d, c.f, sh_n, sh_stride, ch_gu, f4, &m.us)) != cudaSuccess) return e;
  }
  if (ch_dn > 0) {
    if ((e = weight_map(routed + 2 * (nc + ns), c.f, c.d, c.E, c.stride, ch_dn, f4, &m.dr)) != cudaSuccess) return e;
    if ((e = weight_map(sh + 2 * (nc + ns), c.f, c.d, sh_n, sh_stride, ch_dn, f4, &m.ds)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

TcArgs base_args(const Cfg& c, const Ws& ws, const uint8_t* routed, const uint8_t* sh, float* y, long long T) {
  TcArgs a{};
  a.c = c;
  a.ws = ws;
  a.routed = routed;
  a.shared = sh;
  a.y = y;
  a.T = T;
  a.hterms = c.hterms;
  return a;
}

// Map over `rows` activation rows of `row_bytes` E4M3 codes (the terms of x in position order, or of
// h) as {128 bytes, rows, 128-byte chunks}: a box of 128 bytes x n_tile rows x ch chunks is the B
// tiles of one stage of a work group, chunk after chunk (n_tile x 128 bytes each).
cudaError_t rows_map(CUtensorMap* m, const void* base, long long row_bytes, long long rows, int n_tile, int ch) {
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  cuuint64_t gdim[3] = {128, (cuuint64_t)rows, (cuuint64_t)(row_bytes / 128)};
  cuuint64_t gstr[2] = {(cuuint64_t)row_bytes, 128};
  cuuint32_t box[3] = {128, (cuuint32_t)n_tile, (cuuint32_t)ch}, es[3] = {1, 1, 1};
  if (g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), gdim, gstr, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_gateup(const Cfg& c, const Ws& ws, const uint8_t* routed, const uint8_t* shared, float* y,
                          long long T, long long wg_max, cudaStream_t st, cudaEvent_t mid) {
  TcArgs a = base_args(c, ws, routed, shared, y, T);
  a.terms = c.xterms;
  a.n_tile = round16(c.wgt * c.xterms);
  a.xb_tok = c.wgt;
  a.parts = 1;  // the epilogue needs whole sums (splitting items along d measured slower at decode too)
  a.fp4 = c.fp4;
  a.nch = c.d / (c.fp4 ? 256 : 128);
  size_tiles(a, chunks_per_stage(a.nch, 1), c.f / 128);
  if (a.stages < 2) return cudaErrorInvalidConfiguration;
  TcMaps m;
  cudaError_t e = setup(c, routed, shared, a.ch, 0, m, a.shared);
  if (e != cudaSuccess) return e;
  // x terms in position order (c.gx): a work group's B rows are rows pos0 * xterms .. of xp
  CUtensorMap mx = m.gr;
  if (c.gx) {
    if ((e = rows_map(&mx, ws.xp, c.d, T * (c.k + c.S) * c.xterms, a.n_tile, a.ch)) != cudaSuccess) return e;
    a.tma_b = 1;
  }
  e = launch_tc<GATEUP>(a, m.gr, m.ur, m.gs, m.us, mx, wg_max * 2 * (c.f / 128), st);
  if (e == cudaSuccess && mid) e = cudaEventRecord(mid, st);
  return e;
}

cudaError_t launch_down(const Cfg& c, const Ws& ws, const uint8_t* routed, const uint8_t* shared, float* y,
                        long long T, long long wg_max, cudaStream_t st, cudaEvent_t mid, bool combine) {
  TcArgs a = base_args(c, ws, routed, shared, y, T);
  a.terms = c.hterms;
  a.n_tile = round16(c.wgt_dn * c.hterms);
  a.parts = 1;
  a.fp4 = c.fp4;
  a.nch = c.f / (c.fp4 ? 256 : 128);
  size_tiles(a, chunks_per_stage(a.nch, 1), c.d / 128);
  if (a.stages < 2) return cudaErrorInvalidConfiguration;
  TcMaps m;
  cudaError_t e = setup(c, routed, shared, 0, a.ch, m, a.shared);
  if (e != cudaSuccess) return e;
  // E4M3 form: the h terms of a work group's positions are rows pos0 * 3 .. of h, contiguous: one tensor
  // copy of n_tile rows x 128 bytes per chunk (rows past the group's are loaded too; their MMA columns
  // are not read)
  CUtensorMap mh = m.dr;
  if (!c.fp4) {
    if ((e = rows_map(&mh, ws.hq, c.f, T * (c.k + c.S) * c.hterms, a.n_tile, a.ch)) != cudaSuccess) return e;
    a.tma_b = 1;
  }
  e = launch_tc<DOWN>(a, m.dr, m.dr, m.ds, m.ds, mh, wg_max * (c.d / 128), st);
  if (e == cudaSuccess && mid) e = cudaEventRecord(mid, st);
  if (e != cudaSuccess || !combine) return e;
  return launch_combine(c, ws, y, T, st);
}

cudaError_t launch_combine(const Cfg& c, const Ws& ws, float* y, long long T, cudaStream_t st) {
  if (g_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_sms <= 0) g_sms = 1;
  }
  long long blocks = (T * c.d + 255) / 256;
  if (blocks > 8LL * g_sms) blocks = 8LL * g_sms;
  if (c.Sb > 0) return launch_pdl(k_combine<false, true>, dim3((unsigned)blocks), dim3(256), 0, st, c, ws, y, T);
  if (T <= kCombBatchMaxT) return launch_pdl(k_combine<true, false>, dim3((unsigned)blocks), dim3(256), 0, st, c, ws, y, T);
  return launch_pdl(k_combine<false, false>, dim3((unsigned)blocks), dim3(256), 0, st, c, ws, y, T);
}

cudaError_t launch_pack_records(uint8_t* records, long long n_rec, long long stride, int d, int f, int to_device,
                                cudaStream_t st) {
  // a gate/up pair stages two tiles of d/32 scale bytes per row, a down tile one of f/32
  const size_t smem = (size_t)128 * (2 * (d / 32) > f / 32 ? 2 * (d / 32) : f / 32);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_pack_records, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const long long units = n_rec * ((long long)(f / 128) + d / 128);
  if (g_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_sms <= 0) g_sms = 1;
  }
  const long long grid = units < 8LL * g_sms ? units : 8LL * g_sms;
  k_pack_records<<<(unsigned)(grid > 0 ? grid : 1), 256, smem, st>>>(records, n_rec, stride, d, f, to_device);
  return cudaGetLastError();
}

}  // namespace k3
