// la_attn.cu -- attention forward on sm_103a: O = softmax(scale Q K^T) V.
//
// The method is online softmax over key/value tiles ("GPU Kernel for a
// Transformer Layer", section What we learned: a running row max, row sum and
// output accumulator carried across key/value blocks, so the
// [B, H, S_q, S_kv] score matrix is never formed), applied to the attention
// equation of "Shape-Aware Attention" (section Inspiration), with causal and
// key-padding masks.
//
// A work item is NQ query tiles of 128 rows of one (batch, head) against a
// range of 128-key tiles (the whole causal/padded range, or one split of it).
// With no more items than SMs each CTA runs one item; otherwise one CTA per
// SM takes items by ticket (the persistent form).  Roles in a CTA:
//
//   warp 4*NQ   (TMA)      loads Q, then K_j / V_j through an NS-stage ring
//                          of shared-memory buffers (128-byte swizzle), and
//                          in the persistent form draws the items and hands
//                          them to the other warps.  For fp32 (TF32
//                          products, which take K-major operands only) V
//                          comes from its transpose V^T; an fp32 item of one
//                          key tile (one CTA per item) may instead load V
//                          row-major into the idle second stage, and this
//                          warp writes it transposed into the first.
//   warps 4*NQ+1..         tcgen05.mma issuers (one, or one per query tile
//   (MMA)                  where Q sits in tensor memory):  S_t = Q_t K_j^T
//                          into tensor memory, then O_t += P_t V_j with P_t
//                          read straight from tensor memory (A operand in
//                          TMEM).
//   warps 4t..4t+3         softmax of query tile t: thread r owns row r of
//   (softmax, tile t)      S_t (tcgen05.ld 32x32b), applies the mask, keeps
//                          the running max m and sum l in registers, writes
//                          P = exp2(S*scale*log2e - m) back over S (bf16/f16
//                          packed pairs, or tf32), and rescales O_t in tensor
//                          memory when the max grows; finally O_t / l -> HBM.
//                          Where it fits they first copy Q_t into tensor
//                          memory, so that QK^T reads only K from shared
//                          memory.
//
// Half precision D=64 adds a padding warp, so that the TMA and MMA warps
// fill a warpgroup of their own, and moves registers from that warpgroup to
// the softmax warpgroups (setmaxnreg; Cfg::SMR).
//
// The two query tiles ping-pong: while tile 0's softmax runs, the tensor core
// computes PV and the next QK^T of tile 1, and vice versa.  Per tile the MMA
// issue order is PV_t(j) before S_t(j+1), so when the softmax sees S_t(j+1)
// complete, PV_t(j) is complete as well; the O rescale and the P overwrite
// need no other wait.
//
// The max is only moved (and O rescaled) when it grows by more than 2^8; P is
// then bounded by 256 and the final O / l stays exact because both use the
// same stale max.
//
// Every wait is bounded (la_device.cuh); a wait that runs out latches the
// device error word and the CTA winds down, freeing its tensor memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "la_device.cuh"
#include "la_internal.h"

namespace la {
namespace {

template <typename T>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
  static constexpr uint32_t ab = AB_BF16;
  static constexpr bool tf32 = false;
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
};
template <>
struct Elem<__half> {
  static constexpr uint32_t ab = AB_F16;
  static constexpr bool tf32 = false;
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
};
template <>
struct Elem<float> {
  static constexpr uint32_t ab = AB_TF32;
  static constexpr bool tf32 = true;
};

constexpr int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p *= 2;
  return p;
}

// PERS: the persistent form, for launches with more work items than SMs;
// otherwise each CTA runs exactly one item (no item hand-off, and the
// epilogue stages its stores in the dead Q tiles).
template <typename T, int D_, int NQ_, int BN_, int NS_, bool PERS = true>
struct Cfg {
  static constexpr int D = D_, NQ = NQ_, BN = BN_, NS = NS_;
  static constexpr int E = sizeof(T);
  static constexpr int CW = 128 / E;            // elements per 128-byte swizzle row
  static constexpr int NCH = D / CW;            // 128-byte chunks per row of D elements
  static constexpr int Q_CHUNK = kTileM * 128;  // bytes of one chunk of a Q tile
  static constexpr int KV_CHUNK = BN * 128;
  static constexpr int Q_TILE = NCH * Q_CHUNK;
  static constexpr int KV_TILE = NCH * KV_CHUNK;
  // Q as the A operand of QK^T from tensor memory when it fits: the product
  // then reads only K from shared memory (half the operand traffic).
  static constexpr int QCOLS = D * E / 4;                  // 32-bit TMEM columns of one Q row
  static constexpr bool QT = NQ * (BN + D + QCOLS) <= 512;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQ * Q_TILE;
  static constexpr int OFF_V = OFF_K + NS * KV_TILE;
  // Epilogue stores: persistent fp32 stores each thread's 256- or 512-byte
  // row directly (measured 2% faster on fp32 causal S=2048 than through the
  // boxes); the other persistent forms go through 4 KB store boxes per
  // softmax warp, so that each store instruction writes whole 128-byte row
  // segments; the single-item form stages in its dead Q tiles.
  static constexpr bool DIRECT_O = (E == 4) && PERS;
  static constexpr int OFF_STG = OFF_V + NS * KV_TILE;  // epilogue store boxes (PERS, not DIRECT_O)
  static constexpr int OFF_BAR = OFF_STG + (PERS && !DIRECT_O ? NQ * 4 * 4096 : 0);
  // q_full, q_empty, k_full[NS], k_empty[NS], v_full[NS], v_empty[NS], s_full[NQ], p_full[NQ],
  // o_full[NQ], o_free[NQ], mma_done, qt_full, item_full[NR], item_empty[NR]
  static constexpr int NR = 4;  // work items handed from the scheduling thread to the other roles
  static constexpr int NBAR = 2 + 4 * NS + 4 * NQ + 2 + 2 * NR;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // TMEM address, abort flag, then the item ring
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 4 * NR + 1024;  // + slack for 1024-byte alignment
  // per query tile: S (P over it), O, then Q (QT)
  static constexpr int O_COL = BN;
  static constexpr int TILE_COLS = O_COL + D + (QT ? QCOLS : 0);
  static constexpr int TMEM_COLS = pow2_at_least(NQ * TILE_COLS);
  static constexpr int QK_STEPS = D * E / 32;              // one MMA consumes 32 bytes of a row
  static constexpr int PV_ROWS = 32 / E;                   // keys per PV MMA (16, or 8 for tf32)
  static constexpr int PV_STEPS = BN / PV_ROWS;
  // TF32 takes K-major operands only: V then arrives transposed (V^T rows are
  // head dims, keys contiguous) and a V tile is BN*E/128 chunks of D rows.
  static constexpr bool VT = (E == 4);
  static constexpr int VT_CHUNK = D * 128;
  // MMA warps.  With Q in tensor memory, one per query tile, so that one
  // warp's barrier waits and commits overlap the other's MMA issue
  // (measured: fp32 D=64 +5%, bf16 D=64 +3%).  With Q in shared memory one
  // warp, which keeps the strict PV_0, S_0, PV_1, S_1 order (measured: two
  // warps cost bf16 D=128 10%).
  static constexpr int MW = QT ? NQ : 1;
  // One barrier pair per key/value stage (KVM) where measured faster: with Q
  // in tensor memory (fp32 D=64 +3%, bf16 D=64 +7%); bf16 D=128 with its
  // two 64 KB stages needs the key slot back before PV is done (-7%).
  static constexpr bool KVM = QT;
  // Register split (SMR): the block of more than 256 threads is launched at
  // 168 registers a thread; the softmax warpgroups then take R_SOFT and the
  // TMA and MMA warps (with a padding warp, so that they fill a warpgroup)
  // give back to R_REST: 256 x 184 + 128 x 120 = 62464 <= 384 x 168.
  // Measured for half precision D=64 (window B2 H16 S_q4096 S_kv40960
  // 1375 against 1399 us, causal S=4096 133 against 138 us); fp32 D=64 and
  // half precision D=128 measured 1% slower with it, and a larger softmax
  // share spills in the MMA and TMA warps.
  static constexpr bool SMR = (E == 2) && (D == 64) && (NQ == 2);
  static constexpr int R_SOFT = 184, R_REST = 120;
  static constexpr int THREADS_USED = NQ * 128 + 32 + 32 * MW;
  static constexpr int THREADS = SMR ? (THREADS_USED + 127) / 128 * 128 : THREADS_USED;
  static_assert(!SMR || NQ * 128 * R_SOFT + (THREADS - NQ * 128) * R_REST <= THREADS * 168, "register split");
  static constexpr int WARP_TMA = NQ * 4;
  static constexpr int WARP_MMA = NQ * 4 + 1;  // first MMA warp
  static_assert(D % CW == 0, "head dim must fill whole 128-byte rows");
  static_assert(TMEM_COLS <= 512, "tensor memory budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(BN == 64 || BN == 128, "key tile");
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

// TMEM -> registers for a full row of BN fp32 scores.
template <int BN>
__device__ __forceinline__ void load_row(uint32_t taddr, uint32_t (&s)[BN]) {
  if constexpr (BN == 128) {
    tmem_ld_x128(taddr, s);
  } else {
    tmem_ld_x64(taddr, s);
  }
}

// 32 fp32 values -> 32 output elements at dst (16-byte aligned).
template <typename T>
__device__ __forceinline__ void store_out32(T* dst, const float (&v)[32]) {
  if constexpr (Elem<T>::tf32) {
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int i = 0; i < 8; ++i) d4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 w;
      w.x = Elem<T>::pack2(v[8 * i + 0], v[8 * i + 1]);
      w.y = Elem<T>::pack2(v[8 * i + 2], v[8 * i + 3]);
      w.z = Elem<T>::pack2(v[8 * i + 4], v[8 * i + 5]);
      w.w = Elem<T>::pack2(v[8 * i + 6], v[8 * i + 7]);
      d4[i] = w;
    }
  }
}

// Packs 128 bytes of output (32 fp32 or 64 half-precision values) into
// eight 16-byte units; unit u of v.
template <typename T>
__device__ __forceinline__ uint4 pack_unit(const float* v, int u) {
  if constexpr (Elem<T>::tf32) {
    return make_uint4(f2u(v[4 * u]), f2u(v[4 * u + 1]), f2u(v[4 * u + 2]), f2u(v[4 * u + 3]));
  } else {
    uint4 w;
    w.x = Elem<T>::pack2(v[8 * u + 0], v[8 * u + 1]);
    w.y = Elem<T>::pack2(v[8 * u + 2], v[8 * u + 3]);
    w.z = Elem<T>::pack2(v[8 * u + 4], v[8 * u + 5]);
    w.w = Elem<T>::pack2(v[8 * u + 6], v[8 * u + 7]);
    return w;
  }
}

// One work item: the NQ query tiles of query block qblk of head (b, h),
// against key tiles [jb, je_all) (one split of the key range).
struct Item {
  int qblk, b, h, bh, split, kv_lim, jb, je_all;
};

// Causal items are numbered by groups of a.head_group (b, h) pairs, and
// within a group with the query block outermost, the heaviest block (last
// rows) first: handing them out in order is a longest-first schedule whose
// last items are light, while the items running at once read the keys and
// values of a few groups only, which stay in L2.  Non-causal items all weigh
// the same: they are numbered head by head, so that the query blocks of a
// head (which read the same keys and values) run side by side.  Key-range
// splits are innermost.
// je[t] is one past the last key tile of query tile t (jb when it has none).
template <int NQ, int BN>
__device__ __forceinline__ Item decode_item(const AttnArgs& a, int idx, int (&je)[NQ]) {
  Item w;
  int qi;
  if (a.causal) {
    const int per_grp = a.head_group * a.num_qblk * a.splits;
    const int g = idx / per_grp;
    const int bh0 = g * a.head_group;
    const int per_q = min(a.head_group, a.B * a.H - bh0) * a.splits;  // the last group may be short
    const int rem0 = idx - g * per_grp;
    qi = rem0 / per_q;
    const int rem = rem0 - qi * per_q;
    const int pair = rem / a.splits;
    w.bh = bh0 + pair;
    w.split = rem - pair * a.splits;
  } else {
    const int per_bh = a.num_qblk * a.splits;
    w.bh = idx / per_bh;
    const int rem = idx - w.bh * per_bh;
    qi = rem / a.splits;
    w.split = rem - qi * a.splits;
  }
  w.qblk = a.causal ? a.num_qblk - 1 - qi : qi;
  w.b = w.bh / a.H;
  w.h = w.bh - w.b * a.H;
  const int off = a.S_kv - a.S_q;  // query row i is absolute position i + off
  int kv_lim = a.S_kv;
  if (a.kv_len != nullptr) kv_lim = min(kv_lim, max(a.kv_len[w.b], 0));
  w.kv_lim = kv_lim;
  w.jb = w.split * a.tiles_per_split;
  w.je_all = w.jb;
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    const int q_lo = (w.qblk * NQ + t) * kTileM;
    int n = 0;
    if (q_lo < a.S_q) {
      int hi = kv_lim;
      if (a.causal) hi = min(hi, min(q_lo + kTileM - 1, a.S_q - 1) + off + 1);
      n = hi > 0 ? (hi + BN - 1) / BN : 0;
    }
    je[t] = max(w.jb, min(n, w.jb + a.tiles_per_split));
    w.je_all = max(w.je_all, je[t]);
  }
  return w;
}

// V [BN keys, D] -> V^T [D, BN keys] in shared memory.  The source holds
// 128-byte rows of CW head dims (chunk c = dims c*CW.., KV_CHUNK bytes), the
// destination 128-byte rows of CW keys (chunk jc = keys jc*CW.., VT_CHUNK
// bytes), both in the 128-byte swizzle the tensor copies use (16-byte unit u
// of row r at u ^ r%8).  By 4x4 blocks (four 16-byte loads, four 16-byte
// stores): in pass i lane l takes key block 8*(g % NA8) + l%4 + 4*(i & 1) and
// dim block 8*(g / NA8) + l/4 (g = i / 2), so that every load and store
// instruction of the warp touches each of the eight 16-byte bank positions
// exactly four times (no bank conflict).
template <int D, int BN, int CW, int KV_CHUNK, int VT_CHUNK>
__device__ __forceinline__ void transpose_v_tile(uint32_t src, uint32_t dst, int lane) {
  constexpr int NA8 = BN / 32, NB8 = D / 32;
  static_assert(BN % 32 == 0 && D % 32 == 0, "8x8 groups of 4x4 blocks");
#pragma unroll 1
  for (int i = 0; i < 2 * NA8 * NB8; ++i) {
    const int g = i >> 1;
    const int k0 = 4 * (8 * (g % NA8) + (lane & 3) + 4 * (i & 1));
    const int d0 = 4 * (8 * (g / NA8) + (lane >> 2));
    const int c = d0 / CW, u = (d0 % CW) / 4;
    uint32_t e[4][4];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int rk = k0 + rr;
      const uint4 x = lds128(src + c * KV_CHUNK + rk * 128 + ((u ^ (rk & 7)) << 4));
      e[rr][0] = x.x, e[rr][1] = x.y, e[rr][2] = x.z, e[rr][3] = x.w;
    }
    const int jc = k0 / CW, u2 = (k0 % CW) / 4;
#pragma unroll
    for (int dd = 0; dd < 4; ++dd) {
      const int d = d0 + dd;
      sts128(dst + jc * VT_CHUNK + d * 128 + ((u2 ^ (d & 7)) << 4), make_uint4(e[0][dd], e[1][dd], e[2][dd], e[3][dd]));
    }
  }
}

// je[t] for a t not known at compile time, without indexing local memory.
template <int NQ>
__device__ __forceinline__ int sel(const int (&je)[NQ], int t) {
  int v = je[0];
#pragma unroll
  for (int u = 1; u < NQ; ++u)
    if (u == t) v = je[u];
  return v;
}

// The ticket word and the done word each hold a launch tag in their high half
// and a count in their low half.  claim(): once per CTA, before its first
// increment of the word; a word not yet carrying this launch's tag (zero
// after a reset, or whatever a fresh workspace held) is set to (tag, 0) by
// one compare-and-swap.  If that swap fails, another CTA of the launch has
// just claimed the word (nothing else writes it), so one attempt suffices and
// no CTA ever loops on it; increments are then plain atomic adds.
__device__ __forceinline__ void claim(unsigned long long* w, unsigned tag) {
  const unsigned long long cur = atomicAdd(w, 0ull);  // read at the L2, not from a stale line
  if (static_cast<unsigned>(cur >> 32) != tag) atomicCAS(w, cur, static_cast<unsigned long long>(tag) << 32);
}
// Increment of a claimed word: the count before it, or false (and the error
// word latched) if the word does not carry this launch's tag.
__device__ __forceinline__ bool tagged_add(unsigned long long* w, unsigned tag, uint32_t* err, unsigned* before) {
  const unsigned long long old = atomicAdd(w, 1ull);
  if (static_cast<unsigned>(old >> 32) != tag) {
    atomicOr(err, DEVERR_INTERNAL);
    return false;
  }
  *before = static_cast<unsigned>(old);
  return true;
}

// Persistent: one CTA per SM.  CTA c starts with item c; further items come
// by ticket (heaviest first, whichever CTA is free next), ticket t meaning
// item gridDim.x + t.  Barrier phases and the key/value ring continue from
// one item to the next, so an item's loads are issued while the previous
// item finishes.  The ticket word a.sched[0] and the done word a.sched[1]
// live in the caller's workspace, so launches that run at the same time
// (disjoint workspaces) never share them; both carry this launch's tag
// (claim), so a fresh workspace needs no clearing.  Every CTA draws until it
// gets a ticket past the last item, then counts itself done, and the last
// CTA done sets both words to zero, so a replay of the launch from a CUDA
// graph (same tag) claims them afresh and starts again from ticket 0.
template <typename T, int D, int NQ, int BN, int NS, bool PERS>
__global__ void __launch_bounds__(Cfg<T, D, NQ, BN, NS, PERS>::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
  using C = Cfg<T, D, NQ, BN, NS, PERS>;
  constexpr bool TF32 = Elem<T>::tf32;
  // fp32 items of one key tile, one per CTA (a.v_raw): V arrives row-major in
  // the second stage's value buffer, unused with one key tile, and the TMA
  // warp transposes it into the first stage's V^T tile (v_full[1]: the raw
  // tile landed; v_full[0]: V^T written; both unused when keys and values
  // share k_full)
  constexpr bool VRAW_OK = C::VT && C::KVM && !PERS && NS >= 2;
  const bool vraw = VRAW_OK && a.v_raw != 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* q_empty = q_full + 1;  // Q in shared memory: the item's MMAs are done (one commit per MMA warp)
  // With KVM the key and value tiles of a stage share k_full / k_empty (one
  // wait and one commit per key tile; v_full / v_empty unused); otherwise K
  // and V have their own, so that a key slot frees as soon as QK^T is done.
  uint64_t* k_full = q_empty + 1;
  uint64_t* k_empty = k_full + NS;
  uint64_t* v_full = k_empty + NS;
  uint64_t* v_empty = v_full + NS;
  uint64_t* s_full = v_empty + NS;
  uint64_t* p_full = s_full + NQ;
  uint64_t* o_full = p_full + NQ;
  uint64_t* o_free = o_full + NQ;  // O of query tile t read out (one arrive per softmax warp)
  uint64_t* mma_done = o_free + NQ;
  uint64_t* qt_full = mma_done + 1;  // Q copied into tensor memory (one arrive per softmax warp)
  uint64_t* item_full = qt_full + 1;  // ring slot holds the next item (-1: none left)
  uint64_t* item_empty = item_full + C::NR;  // every consumer warp has read the slot
  // the Q shared tiles may take the next item's load once: the copy into
  // tensor memory is done (QT), or the item's MMAs have completed
  uint64_t* q_free = C::QT ? qt_full : q_empty;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* ring = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- set-up ---------------------------------------------------------------
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, C::MW);  // one commit per MMA warp
    for (int s = 0; s < NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], C::MW);  // one commit per MMA warp
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], C::MW);
    }
    for (int t = 0; t < NQ; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);  // one arrive per softmax warp
      mbar_init(&o_full[t], 1);
      mbar_init(&o_free[t], 4);
    }
    mbar_init(mma_done, C::MW);
    mbar_init(qt_full, 4 * NQ);
    for (int r = 0; r < C::NR; ++r) {
      mbar_init(&item_full[r], 1);
      mbar_init(&item_empty[r], C::MW + 4 * NQ);  // MMA warps and softmax warps
    }
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == C::WARP_MMA) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{a.err, abort_flag};
  // The set-up above overlaps the previous grid; nothing before the wait
  // reads or writes global memory the previous grid may touch.  The tensor
  // maps are kernel parameters, so their descriptors are fetched meanwhile.
  // The next grid may be scheduled now: its CTAs take SMs as this grid's
  // retire and wait for all of it before touching memory.
  if (threadIdx.x == 0) pdl_trigger();
  if (warp == C::WARP_TMA && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  pdl_wait();

  const int n_items = a.num_qblk * a.B * a.H * a.splits;
  const int off = a.S_kv - a.S_q;  // query row i is absolute position i + off
  // The next item from the ring (consumer side): -1 when none is left or a
  // wait ran out.  Called by a whole converged warp (softmax) or by lane 0
  // alone (MMA issuers); one arrive per warp frees the slot.
  auto next_item = [&](int& n_taken, bool whole_warp) -> int {
    const int rs = n_taken % C::NR, rr = n_taken / C::NR;
    ++n_taken;
    bool got = mbar_wait(&item_full[rs], rr & 1, ab, SITE_Q_FULL);
    if (whole_warp) got = __all_sync(0xffffffffu, got);
    if (!got) return -1;
    const int idx = ring[rs];
    if (whole_warp) __syncwarp();
    if (lane == 0) mbar_arrive(&item_empty[rs]);
    return idx;
  };

  if (warp == C::WARP_TMA) {
    // ======================= TMA producer ==================================
    if constexpr (C::SMR) setmaxnreg_dec<C::R_REST>();
    int last_k[NS], last_v[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) last_k[s] = last_v[s] = -1;
    int q_last = -1;  // item count of the last Q load issued
    if (lane == 0) {
      const uint64_t pol_q = policy_evict_first();
      // The first item's Q goes out before anything else: after an L2 flush
      // the first instructions of this path miss in the instruction cache,
      // and everything issued ahead of the load delays it.
      bool q_pre = false;
      {
        int je0[NQ];
        const Item w0 = decode_item<NQ, BN>(a, blockIdx.x, je0);
        if (w0.je_all > w0.jb && !a.skip_loads) {
          mbar_arrive_expect_tx(q_full, NQ * C::Q_TILE);
          for (int t = 0; t < NQ; ++t)
            for (int c = 0; c < C::NCH; ++c)
              tma_load_4d(&tm_q, q_full, smem + C::OFF_Q + t * C::Q_TILE + c * C::Q_CHUNK, c * C::CW,
                          (w0.qblk * NQ + t) * kTileM, w0.h, w0.b, pol_q);
          q_pre = true;
          q_last = 0;
        }
      }
      const uint64_t pol_kv = policy_evict_last();
      const int G = gridDim.x;
      // (with no more items than CTAs there is nothing to hand out: no ticket
      // is drawn and the launcher reserves none)
      const bool sched_on = PERS && n_items > G && a.sched != nullptr;
      bool claimed = false;  // this CTA has claimed both words (after its first item's loads went out)
      auto draw = [&]() -> int {
        if (!sched_on) return -1;
        if (!claimed) {
          claim(a.sched, a.sched_gen);
          claim(a.sched + 1, a.sched_gen);
          claimed = true;
        }
        unsigned tk = 0;
        if (!tagged_add(a.sched, a.sched_gen, a.err, &tk)) return -1;
        return tk < static_cast<unsigned>(n_items - G) ? G + static_cast<int>(tk) : -1;
      };
      int it = 0, na = 0, nr = 0;  // key tiles, active items and ring slots so far
      bool ok = true, drawn_last = false, first = true;
#pragma unroll 1
      while (ok) {
        if (!PERS && !first) break;
        int idx = blockIdx.x;  // the first item needs no ticket and no hand-off
        if (!first) {
          idx = draw();
          drawn_last = idx < 0;
          const int rs = nr % C::NR, rr = nr / C::NR;
          ++nr;
          if (rr > 0 && !mbar_wait(&item_empty[rs], (rr - 1) & 1, ab, SITE_Q_FULL)) break;
          ring[rs] = idx;
          mbar_arrive(&item_full[rs]);  // releases the slot write to the waiting warps
          if (idx < 0) break;
        }
        first = false;
        int je[NQ];
        const Item w = decode_item<NQ, BN>(a, idx, je);
        if (w.je_all <= w.jb || a.skip_loads) continue;
        if (q_pre) {
          q_pre = false;  // the first item's Q is already on its way
        } else {
          // the tiles last held item na - 1, whose MMAs (or Q copy) must be done
          if (na >= 1 && !mbar_wait(q_free, (na - 1) & 1, ab, SITE_Q_FULL)) break;
          mbar_arrive_expect_tx(q_full, NQ * C::Q_TILE);
          for (int t = 0; t < NQ; ++t)
            for (int c = 0; c < C::NCH; ++c)
              tma_load_4d(&tm_q, q_full, smem + C::OFF_Q + t * C::Q_TILE + c * C::Q_CHUNK, c * C::CW,
                          (w.qblk * NQ + t) * kTileM, w.h, w.b, pol_q);
          q_last = na;
        }
        for (int j = w.jb; j < w.je_all; ++j, ++it) {
          const int s = it % NS, r = it / NS;
          if (r > 0 && !mbar_wait(&k_empty[s], (r - 1) & 1, ab, SITE_K_EMPTY)) { ok = false; break; }
          mbar_arrive_expect_tx(&k_full[s], (C::KVM && !vraw) ? 2 * C::KV_TILE : C::KV_TILE);
          for (int c = 0; c < C::NCH; ++c)
            tma_load_4d(&tm_k, &k_full[s], smem + C::OFF_K + s * C::KV_TILE + c * C::KV_CHUNK, c * C::CW,
                        j * BN, w.h, w.b, pol_kv);
          last_k[s] = r;
          uint64_t* vbar = C::KVM ? &k_full[s] : &v_full[s];
          if constexpr (!C::KVM) {
            if (r > 0 && !mbar_wait(&v_empty[s], (r - 1) & 1, ab, SITE_V_EMPTY)) { ok = false; break; }
            mbar_arrive_expect_tx(vbar, C::KV_TILE);
          }
          if constexpr (C::VT) {
            if (vraw) {  // the item's one value tile, row-major, into the second stage's buffer
              mbar_arrive_expect_tx(&v_full[1], C::KV_TILE);
              for (int c = 0; c < C::NCH; ++c)
                tma_load_4d(&tm_v, &v_full[1], smem + C::OFF_V + C::KV_TILE + c * C::KV_CHUNK, c * C::CW, j * BN,
                            w.h, w.b, pol_kv);
              last_v[1] = 0;
            } else {
              for (int c = 0; c < BN / C::CW; ++c)
                tma_load_4d(&tm_v, vbar, smem + C::OFF_V + s * C::KV_TILE + c * C::VT_CHUNK, j * BN + c * C::CW,
                            0, w.h, w.b, pol_kv);
            }
          } else {
            for (int c = 0; c < C::NCH; ++c)
              tma_load_4d(&tm_v, vbar, smem + C::OFF_V + s * C::KV_TILE + c * C::KV_CHUNK, c * C::CW, j * BN,
                          w.h, w.b, pol_kv);
          }
          if constexpr (!C::KVM) last_v[s] = r;
        }
        ++na;
      }
      // a CTA that stopped early still draws until the end of the items, so
      // that every CTA ends with a ticket past the last item
      if (PERS && !drawn_last)
        while (draw() >= 0) {
        }
      // The last CTA done drawing returns both words to zero (the fences
      // order every CTA's last draw before its done count, and the count
      // before the reset).
      if (sched_on) {
        if (!claimed) {  // (every path above draws at least once; kept for safety)
          claim(a.sched, a.sched_gen);
          claim(a.sched + 1, a.sched_gen);
        }
        __threadfence();
        unsigned done_before = 0;
        if (tagged_add(a.sched + 1, a.sched_gen, a.err, &done_before) && done_before == static_cast<unsigned>(G - 1)) {
          __threadfence();
          atomicExch(a.sched, 0ull);
          atomicExch(a.sched + 1, 0ull);
        }
      }
    }
    __syncwarp();
    if constexpr (VRAW_OK) {
      // the raw tile (second stage's value buffer) into the first stage's V^T tile
      if (vraw && __shfl_sync(0xffffffffu, last_v[1], 0) == 0 &&
          __all_sync(0xffffffffu, mbar_wait(&v_full[1], 0, ab, SITE_V_FULL))) {
        transpose_v_tile<D, BN, C::CW, C::KV_CHUNK, C::VT_CHUNK>(smem_u32(smem + C::OFF_V + C::KV_TILE),
                                                                smem_u32(smem + C::OFF_V), lane);
        fence_proxy_async_smem();  // the PV products read the tile through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(&v_full[0]);
      }
      __syncwarp();
    }
    __syncthreads();  // teardown rendezvous
    if (lane == 0 && *abort_flag) {
      // let the copies still in flight land before the CTA's shared memory goes away
      if (q_last >= 0) mbar_wait_teardown(q_full, q_last & 1);
      for (int s = 0; s < NS; ++s) {
        if (last_k[s] >= 0) mbar_wait_teardown(&k_full[s], last_k[s] & 1);
        if (last_v[s] >= 0) mbar_wait_teardown(&v_full[s], last_v[s] & 1);
      }
    }
    __syncwarp();
  } else if (warp >= C::WARP_MMA + C::MW) {
    // padding warp of the register split: gives its registers back and
    // joins the teardown rendezvous
    if constexpr (C::SMR) setmaxnreg_dec<C::R_REST>();
    __syncthreads();
  } else if (warp >= C::WARP_MMA) {
    // ======================= MMA issuers ===================================
    if constexpr (C::SMR) setmaxnreg_dec<C::R_REST>();
    // MMA warp m issues for query tiles t = m, m + MW, ...  Step j issues
    // PV(j) and S(j+1).  With KVM, V(j) arrived with K(j) (waited for before
    // S(j)), stage j+1 is waited for before S(j+1), and stage j is freed at
    // the end of the step (its K was last read by S(j), its V by PV(j)).
    // Otherwise V(j) is waited for before PV(j), K(j+1) before S(j+1), and the
    // V slot of j and the K slot of j+1 are freed at the end of the step.
    // Every MMA warp waits for and frees every slot use exactly once (the
    // empty barriers count MW commits), so no warp can run a phase ahead of
    // another.  An item's first PV into O waits until the previous item's O
    // has been read out (o_free).
    const int m = warp - C::WARP_MMA;
    // The whole warp runs the loop (barrier waits by every lane, counters kept
    // by every lane, so the MMA operands are warp-uniform); one elected lane
    // issues each group of MMAs and its commit.
    constexpr unsigned FULL = 0xffffffffu;
    {
      const uint32_t idesc_qk = idesc_make(Elem<T>::ab, kTileM, BN, false, false);
      const uint32_t idesc_pv = idesc_make(Elem<T>::ab, kTileM, D, false, !C::VT);
      // Shared-memory descriptors of the tile bases; the start address field
      // holds address >> 4 and every address here stays below 2^18, so a byte
      // offset is added to a descriptor as (offset >> 4).
      const uint64_t dQ = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
      const uint64_t dK = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);
      const uint64_t dV = C::VT ? sdesc_sw128(smem_u32(smem + C::OFF_V), 16, 1024)
                                : sdesc_sw128(smem_u32(smem + C::OFF_V), C::KV_CHUNK, 1024);
      // S_t = Q_t K^T into the S columns of query tile t (K tile at descriptor bK)
      auto issue_s = [&](int t, uint64_t bK) {
        const uint64_t a0 = dQ + ((t * C::Q_TILE) >> 4);
#pragma unroll
        for (int kk = 0; kk < C::QK_STEPS; ++kk) {
          const uint32_t off_q = ((kk >> 2) * C::Q_CHUNK + (kk & 3) * 32) >> 4;
          const uint32_t off_k = ((kk >> 2) * C::KV_CHUNK + (kk & 3) * 32) >> 4;
          if constexpr (C::QT)
            mma_ts<TF32>(tmem + t * C::TILE_COLS, tmem + t * C::TILE_COLS + C::O_COL + D + kk * 8, bK + off_k, idesc_qk,
                         kk > 0 ? 1u : 0u);
          else
            mma_ss<TF32>(tmem + t * C::TILE_COLS, a0 + off_q, bK + off_k, idesc_qk, kk > 0 ? 1u : 0u);
        }
      };
      auto wait_all = [&](uint64_t* bar, uint32_t parity, uint32_t site) -> bool {
        return __all_sync(FULL, mbar_wait(bar, parity, ab, site));
      };
      constexpr int TPW = NQ / C::MW;  // query tiles per MMA warp: t = m + tt * MW
      int it = 0, na = 0;
      int sp[TPW], oc[TPW];  // per own query tile: S/P tiles and outputs so far (barrier phases)
#pragma unroll
      for (int tt = 0; tt < TPW; ++tt) sp[tt] = oc[tt] = 0;
      bool ok = true;
      int taken = -1;
#pragma unroll 1
      while (ok) {
        if (!PERS && taken >= 0) break;
        const int idx = taken < 0 ? static_cast<int>(blockIdx.x) : next_item(taken, true);
        if (taken < 0) taken = 0;
        if (idx < 0) break;
        int je[NQ];
        const Item w = decode_item<NQ, BN>(a, idx, je);
        if (w.je_all <= w.jb) continue;
        ok = wait_all(C::QT ? qt_full : &q_full[0], na & 1, SITE_Q_FULL) &&
             wait_all(&k_full[it % NS], (it / NS) & 1, SITE_K_FULL);
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int tt = 0; tt < TPW; ++tt) {
            const int t = m + tt * C::MW;
            if (sel(je, t) > w.jb) {
              issue_s(t, dK + (((it % NS) * C::KV_TILE) >> 4));
              mma_commit(&s_full[t]);
            }
          }
          if constexpr (!C::KVM) mma_commit(&k_empty[it % NS]);
        }
        __syncwarp();
        for (int j = w.jb; ok && j < w.je_all; ++j) {
          const int i = it + (j - w.jb);
          const int s = i % NS, r = i / NS;
          const int sn = (i + 1) % NS, rn = (i + 1) / NS;
          const uint64_t bV = dV + ((s * C::KV_TILE) >> 4);
          const uint64_t bK = dK + ((sn * C::KV_TILE) >> 4);
          bool v_ready = C::KVM && !vraw, k_next = false;
#pragma unroll
          for (int tt = 0; tt < TPW; ++tt) {
            const int t = m + tt * C::MW;
            const int je_t = sel(je, t);
            if (!ok || j >= je_t) continue;
            ok = wait_all(&p_full[t], sp[tt] & 1, SITE_P_FULL);
            if (ok && j == w.jb && oc[tt] > 0) ok = wait_all(&o_free[t], (oc[tt] - 1) & 1, SITE_O_FULL);
            if (ok && !v_ready) ok = v_ready = wait_all(&v_full[s], r & 1, SITE_V_FULL);
            if (!ok) continue;
            tc_fence_after();
            ++sp[tt];
            const bool more = j + 1 < je_t;
            if (elect_one()) {
              // O_t += P_t V: P from tensor memory; V MN-major (rows = keys), or for
              // TF32 the K-major V^T tile (rows = head dims, 8 keys = 32 bytes a step)
              const uint32_t d_o = tmem + t * C::TILE_COLS + C::O_COL;
              const uint32_t p_t = tmem + t * C::TILE_COLS;  // P over S
#pragma unroll
              for (int kk = 0; kk < C::PV_STEPS; ++kk) {
                const uint32_t off = C::VT ? ((kk >> 2) * C::VT_CHUNK + (kk & 3) * 32) >> 4
                                           : (kk * C::PV_ROWS * 128) >> 4;
                mma_ts<TF32>(d_o, p_t + kk * 8, bV + off, idesc_pv, (j > w.jb || kk > 0) ? 1u : 0u);
              }
              if (!more) mma_commit(&o_full[t]);
            }
            __syncwarp();
            if (more) {
              if (!k_next) {
                ok = k_next = wait_all(&k_full[sn], rn & 1, SITE_K_FULL);
                if (!ok) continue;
                tc_fence_after();
              }
              if (elect_one()) {
                issue_s(t, bK);
                mma_commit(&s_full[t]);
              }
              __syncwarp();
            } else {
              ++oc[tt];
            }
          }
          if (!ok) break;
          if constexpr (C::KVM) {
            // stage j+1 must be seen full by every MMA warp before stage j is
            // freed, which keeps each warp's waits in phase order
            if (j + 1 < w.je_all && !k_next) ok = wait_all(&k_full[sn], rn & 1, SITE_K_FULL);
            if (!ok) break;
            if (elect_one()) mma_commit(&k_empty[s]);
            __syncwarp();
          } else {
            if (!v_ready) ok = wait_all(&v_full[s], r & 1, SITE_V_FULL);
            if (!ok) break;
            if (elect_one()) mma_commit(&v_empty[s]);
            __syncwarp();
            if (j + 1 < w.je_all) {
              if (!k_next) ok = wait_all(&k_full[sn], rn & 1, SITE_K_FULL);
              if (!ok) break;
              if (elect_one()) mma_commit(&k_empty[sn]);
              __syncwarp();
            }
          }
        }
        if (!ok) break;
        // Q in shared memory: free for the next item's load once this item's
        // last QK^T (issued above) has completed
        if constexpr (!C::QT) {
          if (elect_one()) mma_commit(&q_empty[0]);
          __syncwarp();
        }
        it += w.je_all - w.jb;
        ++na;
      }
    }
    __syncwarp();
    __syncthreads();  // teardown rendezvous
    if (*abort_flag) {
      if (elect_one()) {  // the lane that issued this warp's MMAs
        mma_commit(mma_done);  // fires once every MMA warp's issued MMAs have finished
        mbar_wait_teardown(mma_done, 0);
      }
      __syncwarp();
    }
    if (warp == C::WARP_MMA) {  // the warp that allocated
      tc_fence_after();
      tmem_dealloc(tmem, C::TMEM_COLS);
    }
  } else {
    // ======================= softmax of query tile t ========================
    if constexpr (C::SMR) setmaxnreg_inc<C::R_SOFT>();
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t tS = tmem + (static_cast<uint32_t>(wq * 32) << 16) + t * C::TILE_COLS;
    const uint32_t tO = tS + C::O_COL;
    int sc = 0, oc = 0, na = 0;  // S tiles, outputs and Q copies so far (barrier phases)
    bool ok = true;
    // Copy this thread's Q row of item idx (TF32-rounded by the load for
    // fp32; packed pairs for bf16/fp16) from the swizzled shared tile into
    // tensor-memory lane `row`, the layout an A operand takes there.  The
    // previous item's QK^T products of this tile, which read the old Q there,
    // all completed before its last scores were read.
    auto copy_q = [&](int idx) -> bool {
      int je[NQ];
      const Item w = decode_item<NQ, BN>(a, idx, je);
      if (!C::QT || w.je_all <= w.jb) return true;
      bool good = __all_sync(0xffffffffu, mbar_wait(q_full, na & 1, ab, SITE_Q_FULL));
      if (good) {
        const uint32_t qs = smem_u32(smem + C::OFF_Q + t * C::Q_TILE) + row * 128;
#pragma unroll
        for (int c = 0; c < C::NCH; ++c) {
          uint32_t wv[32];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 x = lds128(qs + c * C::Q_CHUNK + ((u ^ (row & 7)) << 4));
            wv[4 * u] = x.x, wv[4 * u + 1] = x.y, wv[4 * u + 2] = x.z, wv[4 * u + 3] = x.w;
          }
          tmem_st_x32(tO + D + c * 32, wv);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(qt_full);
      ++na;
      return good;
    };
    int taken = 0;
    int idx = blockIdx.x;  // the first item needs no hand-off
    ok = copy_q(idx);
#pragma unroll 1
    while (ok) {
      int q_lo, kv_lim, jb, je_t;
      {
        int je[NQ];
        const Item w = decode_item<NQ, BN>(a, idx, je);
        q_lo = (w.qblk * NQ + t) * kTileM;
        kv_lim = w.kv_lim;
        jb = w.jb;
        je_t = jb;  // this tile's key-tile end, kept in a register
#pragma unroll
        for (int u = 0; u < NQ; ++u)
          if (u == t) je_t = je[u];
      }
      const int q_row = q_lo + row;
      float m_run = -INFINITY;  // running max, in log2 units of the scaled scores
      float l = 0.f;            // running sum of P
      for (int j = jb; j < je_t; ++j) {
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[t], sc & 1, ab, SITE_S_FULL));
        if (!ok) break;
        ++sc;
        tc_fence_after();
        uint32_t s[BN];
        load_row<BN>(tS, s);
        const int kv0 = j * BN;
        if (kv0 + BN > kv_lim || (a.causal && kv0 + BN - 1 > q_lo + off)) {
          int lim = kv_lim;
          if (a.causal) lim = min(lim, q_row + off + 1);
          lim -= kv0;
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c >= lim) s[c] = f2u(-INFINITY);
        }
        // row max: 8 independent partial maxima, each folding in two columns
        // per three-input max, then a tree (no 128-long dependency chain)
        float mxa[8];
#pragma unroll
        for (int kq = 0; kq < 8; ++kq) mxa[kq] = fmaxf(u2f(s[kq]), u2f(s[8 + kq]));
#pragma unroll
        for (int c = 16; c < BN; c += 16)
#pragma unroll
          for (int kq = 0; kq < 8; ++kq) mxa[kq] = fmax3(mxa[kq], u2f(s[c + kq]), u2f(s[c + 8 + kq]));
        const float mx = fmax3(fmax3(mxa[0], mxa[1], mxa[2]), fmax3(mxa[3], mxa[4], mxa[5]), fmaxf(mxa[6], mxa[7]));
        const float m_new = fmaxf(m_run, mx * a.sl2);
        const bool grow = m_new > m_run + 8.0f;
        float alpha = 1.f;
        if (grow) {
          alpha = ex2_approx(m_run - m_new);  // 0 on the first visible key
          l *= alpha;
          m_run = m_new;
        }
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        float rsa[8];  // row sum: 8 independent partial sums
#pragma unroll
        for (int kq = 0; kq < 8; ++kq) rsa[kq] = 0.f;
        // P by halves of 64 columns.  TF32: each half is stored to tensor
        // memory as soon as it is formed (over S, whose values are all in
        // registers by now), formed in place in s[] (a word goes to a slot
        // already read).  TF32 rounds to
        // nearest (ties away) by adding half a TF32 ulp to the bit pattern:
        // the kind::tf32 product reads only the top 19 bits of each 32-bit
        // element, P >= 0 and finite, so a carry into the exponent is the
        // correct rounding (a conversion instruction per element measured
        // ~1000 cycles a row).
#pragma unroll
        for (int h = 0; h < BN; h += 64) {
#pragma unroll
          for (int c = h; c < h + 64; c += 2) {
            // exponent arguments and partial sums two columns per instruction
            float x0, x1;
            fma2(x0, x1, u2f(s[c]), u2f(s[c + 1]), a.sl2, a.sl2, -m_use, -m_use);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            float& r0 = rsa[c & 7];
            float& r1 = rsa[(c & 7) + 1];
            add2(r0, r1, r0, r1, p0, p1);
            if constexpr (TF32) {
              s[c] = f2u(p0) + 0x1000u;
              s[c + 1] = f2u(p1) + 0x1000u;
            } else {
              s[c] = f2u(p0);
              s[c + 1] = f2u(p1);
            }
          }
          if constexpr (TF32) {
            if (h == 0) tmem_st_x64_at<0>(tS, s);
            else tmem_st_x64_at<(BN > 64 ? 64 : 0)>(tS + 64, s);
          }
        }
        if constexpr (!TF32) {
          // half precision over S: packed once the whole row is formed (by
          // halves this form measured spills)
          uint32_t pk[BN / 2];
#pragma unroll
          for (int c = 0; c < BN / 2; ++c) pk[c] = Elem<T>::pack2(u2f(s[2 * c]), u2f(s[2 * c + 1]));
          if constexpr (BN == 128)
            tmem_st_x64(tS, pk);
          else
            tmem_st_x32(tS, pk);
        }
        {
          float a0, a1, b0, b1;
          add2(a0, a1, rsa[0], rsa[1], rsa[2], rsa[3]);
          add2(b0, b1, rsa[4], rsa[5], rsa[6], rsa[7]);
          add2(a0, a1, a0, a1, b0, b1);
          l += a0 + a1;
        }
        // O was produced by PV of earlier tiles: rescale it to the new max.  The
        // tensor-memory loads/stores are warp-collective, so the warp rescales
        // together when any of its rows grew (alpha is 1 for the others).
        if (__any_sync(0xffffffffu, grow) && j > jb) {
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tmem_ld_x32(tO + c0, o);
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = f2u(u2f(o[c]) * alpha);
            tmem_st_x32(tO + c0, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[t]);
      }
      if (!ok) break;
      // The next item's Q goes into tensor memory before this item's output
      // is read out, so that its first QK^T runs during this epilogue.
      const int next = PERS ? next_item(taken, true) : -1;
      if (next >= 0) ok = copy_q(next);
      if (!ok) break;
      const bool has_o = je_t > jb;
      if (has_o) {
        ok = __all_sync(0xffffffffu, mbar_wait(&o_full[t], oc & 1, ab, SITE_O_FULL));
        if (!ok) break;
        ++oc;
        tc_fence_after();
      }
      const bool row_ok = q_row < a.S_q;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      int je_unused[NQ];
      const Item w = decode_item<NQ, BN>(a, idx, je_unused);  // again, for the epilogue
      if (a.part_o != nullptr) {
        // split partial: O / l of this split and its log2-sum-exp
        float* prow = a.part_o + ((static_cast<size_t>(w.split) * a.B * a.H + w.bh) * a.S_q + q_row) * D;
        if (has_o) {
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tmem_ld_x32(tO + c0, o);
            float v[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = u2f(o[c]) * inv;
            if (row_ok && LA_IN_BOUNDS(prow - a.part_o + c0, 32, a.part_elems, a.err))
              store_out32<float>(prow + c0, v);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&o_free[t]);
        } else if (row_ok) {
          const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int c0 = 0; c0 < D; c0 += 4)
            if (LA_IN_BOUNDS(prow - a.part_o + c0, 4, a.part_elems, a.err)) *reinterpret_cast<float4*>(prow + c0) = z;
        }
        if (row_ok && LA_IN_BOUNDS((prow - a.part_o) / D, 1, a.part_elems / D, a.err))
          a.part_lse[(static_cast<size_t>(w.split) * a.B * a.H + w.bh) * a.S_q + q_row] =
              l > 0.f ? m_run + __log2f(l) : -INFINITY;
      } else if (has_o && C::DIRECT_O) {
        T* drow = reinterpret_cast<T*>(a.o) + w.b * a.o_sb + w.h * a.o_sh + static_cast<long long>(q_row) * a.o_ss;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld_x32(tO + c0, o);
          float v[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = u2f(o[c]) * inv;
          if (c0 + 32 >= D) {  // O read out: the next item's PV may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[t]);
          }
          if (row_ok && LA_IN_BOUNDS(drow - reinterpret_cast<T*>(a.o) + c0, 32, a.o_elems, a.err))
            store_out32<T>(drow + c0, v);
        }
      } else if (has_o) {
        // Through shared memory, so that each store instruction writes whole
        // 128-byte row segments (four rows of the warp per instruction).
        // this warp's 4 KB store box (single-item form: a quarter of the query
        // tile's Q buffer, dead since every QK^T of the tile completed)
        const uint32_t stg =
            smem_u32(smem + (PERS ? C::OFF_STG + (t * 4 + wq) * 4096 : C::OFF_Q + t * C::Q_TILE + wq * 4096));
        const int sub = lane >> 3, unit = lane & 7;
        T* dst = reinterpret_cast<T*>(a.o) + w.b * a.o_sb + w.h * a.o_sh + unit * C::CW / 8;
        const int r0 = q_lo + wq * 32;  // query row of lane 0
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += C::CW) {
          float v[C::CW];
#pragma unroll
          for (int hh = 0; hh < C::CW / 32; ++hh) {
            uint32_t o[32];
            tmem_ld_x32(tO + c0 + 32 * hh, o);
#pragma unroll
            for (int c = 0; c < 32; ++c) v[32 * hh + c] = u2f(o[c]) * inv;
          }
          if (c0 + C::CW >= D) {  // O read out: the next item's PV may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[t]);
          }
          __syncwarp();  // the previous chunk's reads of the buffer are done
#pragma unroll
          for (int u = 0; u < 8; ++u) sts128(stg + lane * 128 + ((u ^ (lane & 7)) << 4), pack_unit<T>(v, u));
          __syncwarp();
          uint4 wv[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {  // row 4i + sub of the warp, this lane's 16-byte unit
            const int r = 4 * i + sub;
            wv[i] = lds128(stg + r * 128 + ((unit ^ (r & 7)) << 4));
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = r0 + 4 * i + sub;
            if (rr < a.S_q && LA_IN_BOUNDS(dst - reinterpret_cast<T*>(a.o) + static_cast<long long>(rr) * a.o_ss + c0,
                                           C::CW / 8, a.o_elems, a.err))
              *reinterpret_cast<uint4*>(dst + static_cast<long long>(rr) * a.o_ss + c0) = wv[i];
          }
        }
      } else {
        // no visible key for any row of this tile: zeros
        T* dst = reinterpret_cast<T*>(a.o) + w.b * a.o_sb + w.h * a.o_sh + static_cast<long long>(q_row) * a.o_ss;
        float v[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] = 0.f;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32)
          if (row_ok && LA_IN_BOUNDS(dst - reinterpret_cast<T*>(a.o) + c0, 32, a.o_elems, a.err))
            store_out32<T>(dst + c0, v);
      }
      if (next < 0) break;
      idx = next;
    }
    __syncthreads();  // teardown rendezvous
  }
}

template <typename T, int D, int NQ, int BN, int NS, bool PERS>
cudaError_t launch_form(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& b,
                        int grid, cudaStream_t st) {
  using C = Cfg<T, D, NQ, BN, NS, PERS>;
  auto kern = attn_fwd_kernel<T, D, NQ, BN, NS, PERS>;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if constexpr (C::SMR) {
      // the register split must fit in what the block is launched with
      // (otherwise the softmax warps' increase would never be granted)
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      if (fa.numRegs * C::THREADS < NQ * 128 * C::R_SOFT + (C::THREADS - NQ * 128) * C::R_REST)
        return cudaErrorInvalidConfiguration;
    }
    configured[dev] = true;
  }
  return launch_pdl("attn_fwd_kernel", kern, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, st, tq, tk, tv, b);
}

// One CTA per item when the items fit on the SMs at once, or when there are
// no ticket words (a launch without workspace for them); otherwise the
// persistent form on every SM, drawing items by ticket.
template <typename T, int D, int NQ, int BN, int NS>
cudaError_t launch_one(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a,
                       int splits, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long items = static_cast<long long>(a.num_qblk) * a.B * a.H * splits;
  if (items == 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  AttnArgs b = a;
  b.splits = splits;
  if (items <= sms || a.sched == nullptr)
    return launch_form<T, D, NQ, BN, NS, false>(tq, tk, tv, b, static_cast<int>(items), st);
  return launch_form<T, D, NQ, BN, NS, true>(tq, tk, tv, b, sms, st);
}

}  // namespace

// Launch shapes per (dtype, D): query rows per CTA = 128 * NQ, key tile BN,
// stages NS; chosen so Q + NS stages of K and V fit in 227 KB of shared memory
// and the S|P and O columns of the NQ tiles fit in 512 TMEM columns.
bool attn_shape(la_dtype dt, int D, AttnShape* s) {
  const int e = dt == LA_F32 ? 4 : 2;
  if (D != 64 && D != 128) return false;
  if (dt != LA_F32 && dt != LA_BF16 && dt != LA_F16) return false;
  const bool single = (dt == LA_F32 && D == 128);
  s->rows_per_cta = single ? 128 : 256;
  s->block_n = single ? 64 : 128;
  s->box_q_rows = kTileM;
  s->box_kv_rows = s->block_n;
  s->box_cols = 128 / e;
  return true;
}

cudaError_t launch_attn(la_dtype dt, int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const AttnArgs& a, int splits, cudaStream_t st) {
  switch (dt) {
    case LA_BF16:
      return D == 64 ? launch_one<__nv_bfloat16, 64, 2, 128, 3>(tq, tk, tv, a, splits, st)
                     : launch_one<__nv_bfloat16, 128, 2, 128, 2>(tq, tk, tv, a, splits, st);
    case LA_F16:
      return D == 64 ? launch_one<__half, 64, 2, 128, 3>(tq, tk, tv, a, splits, st)
                     : launch_one<__half, 128, 2, 128, 2>(tq, tk, tv, a, splits, st);
    case LA_F32:
      return D == 64 ? launch_one<float, 64, 2, 128, 2>(tq, tk, tv, a, splits, st)
                     : launch_one<float, 128, 1, 64, 2>(tq, tk, tv, a, splits, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace la
