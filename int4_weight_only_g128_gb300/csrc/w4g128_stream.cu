// The weight-streaming kernels: y_i = x_i . dequant(W_i) for a list of
// int4-g128 matrices -- M = 1 decode and the M <= 16 verify alike on the
// warp-level MMA, so that a row's bits do not depend on M -- and the optional
// residual add + RMS norm the product feeds.
//
// Design (sm_103a, one GPU):
//  * The work is a flat list of items (matrix, 64-column quad, segment of 4
//    groups = 512 rows).  A persistent grid gives each warp a contiguous,
//    balanced range of items ("stream-K").  Segment boundaries are fixed by
//    the shape alone, and every output is the left fold, over segments in
//    order, of fixed-order segment sums -- so y depends on neither the grid,
//    the SM count nor which other matrices share the call.
//  * Each warp streams its chunks (one group x one quad = up to 4 adjacent
//    blocks of 1088 bytes, plus that group's activation package) through a
//    private ring of shared-memory slots filled by 1-D TMA bulk copies
//    (cp.async.bulk) and completed on per-slot mbarriers.  Within a matrix a
//    warp's range is one sequential byte stream.  Warps never wait on each
//    other while streaming (at M = 1 a CTA's warps meet once, at its end).
//  * A quad owned wholly by one warp is written straight to y.  For a quad
//    split between warps every segment sum goes to its own fp32 partial slot
//    (the warp holding the quad's first segments stores their left fold as
//    one slot), and the slots are folded in segment order:
//      - M = 1: each warp takes the tickets of its (at most two) split quads
//        after its stream; the CTA holding a quad's last ticket folds it with
//        all its threads once its warps are done -- no warp stalls mid-stream;
//      - M >= 2: by a reduce kernel launched right behind the streaming
//        kernel (programmatic dependent launch), since 64*M outputs per quad
//        would tie up the SMs that finish last: one CTA per quad pulling a
//        split quad's slots into shared memory with bulk copies, or, for
//        calls with many more quads (mostly owned) than that grid holds at
//        once, one CTA per streaming warp folding the quad that warp's range
//        starts in when the quad began in the warp before.
//  * A small prep kernel (launched first; the streaming kernel overlaps it by
//    programmatic dependent launch) turns x into per-group packages in the
//    order the lanes consume them, with the group sums the factorised
//    dequantisation needs, and clears the status word and the tickets.
//    Every kernel of a call is a programmatic dependent launch, the prep
//    kernel too (behind whatever precedes it; it waits for that to finish
//    before it touches anything), so a call's launches overlap the previous
//    call's tail.
//  * Kernel parameters are read at fixed offsets where possible: a lookup in
//    the matrix table with a computed index is an L2 round trip whenever it
//    misses the constant cache, and on the critical path those add up.
//
// Dequantisation uses the factorised form of w = min + q*scale over a group g:
//     sum_{k in g} x_k w_kn = scale_gn * sum_k x_k q_kn + min_gn * X_g,
//     X_g = sum_{k in g} x_k
// (Token Rush README, "Quantization": 128 weights per bf16 scale and minimum).
// Codes become fp16 values with one LOP3 per pair (a magic-number
// conversion): with the fp16 pattern of 1024 OR-ed in, a nibble at bits 0..3
// of a 16-bit half reads as 1024 + q and a nibble at bits 4..7 as 1024 + 16q,
// so a packed word needs one shift and four LOP3s (bf16, whose mantissa has
// only 7 bits, would need three shifts).  Of each lane's four pairs, the two
// of column r come out as 1024 + q and the two of column r + 8 as 1024 + 16q.
// The activations enter as fp16 too: the prep kernel scales each (group, row)
// of x by a power of two 2^s that puts its largest magnitude in [2^14, 2^15)
// (exact for every value within 2^29 of that largest one), so every product
// x' (1024 + q) is exact in fp32.  With f = 2^-s and X_g the true sum of x,
//     column r:     scale * f * S_g + (min - 1024 scale) * X_g,
//     column r + 8: (scale / 16) * f * S_g + (min - 64 scale) * X_g,
// where S_g is the fp32 sum of x' times the converted code.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "w4g128_internal.h"
#include "w4g128_ptx.cuh"

namespace w4g128 {
namespace {

// ----------------------------------------------------------------- modes

enum Mode : int {
  kMMA = 1,  // 2 <= M <= 8, warp MMA m16n8k16 f16 -> f32 with the weights as the 16-row operand
  kMMA1 = 2, // M = 1: the warp MMA, every B column carrying the one x row
  kMMA16 = 3, // 9 <= M <= 16: the warp MMA, two 8-row x tiles per dequantised weight fragment
};

// The modes that carry p.M x rows through the MMA (and fold in the reduce kernel).
template <int MODE>
__host__ __device__ constexpr bool multi_row() { return MODE == kMMA || MODE == kMMA16; }

#ifndef W4G128_WARPS_PER_CTA
#define W4G128_WARPS_PER_CTA 16
#endif
#ifndef W4G128_RING_DEPTH
#define W4G128_RING_DEPTH 2
#endif
constexpr int kNW = W4G128_WARPS_PER_CTA;  // warps per CTA
constexpr int kDepth = W4G128_RING_DEPTH;  // ring slots per warp

// ----------------------------------------------------------------- debug checks

// Built with -DW4G128_DEBUG, the kernels check the index of every global
// access they derive from the schedule (weight and package copies, x
// staging, partial slots, tickets, y) against its buffer; a check that fails
// records W4G128_ERR_INTERNAL in the status word and the access is skipped
// (a skipped copy still completes its ring slot, so nothing waits for it).
// Nothing traps.  Release builds compile the checks away.
#ifdef W4G128_DEBUG
constexpr bool kDebug = true;
#else
constexpr bool kDebug = false;
#endif

// cond, or (debug builds) false after recording the failure in a 32-bit
// status word (the prep-kernel path's).
__device__ __forceinline__ bool dbg_ok(unsigned* status, bool cond) {
  if constexpr (kDebug) {
    if (!cond) atomicCAS(status, 0u, static_cast<unsigned>(W4G128_ERR_INTERNAL));
    return cond;
  } else {
    return true;
  }
}

// Completes one arrival on an mbarrier without a copy (a skipped copy's slot).
__device__ __forceinline__ void mbar_arrive_plain(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bytes of the packed form of a K x N matrix.
__host__ __device__ inline long long packed_bytes_of(int K, int N) {
  return static_cast<long long>(N / kTileN) * (K / kGroup) * kBlockBytes;
}

// Activation package per group: rows x 4 lane classes c x (16 fp16-pair
// words + 4 unused) = rows x 320 bytes, then per row m the pair
// (X_g[m], f[m]) as fp32.  Row (m, c) word 2i holds x'[m][k0+2c],
// x'[m][k0+2c+1] and word 2i+1 holds x'[m][k0+2c+8], x'[m][k0+2c+9] for
// k0 = 128g + 16i: exactly the fp16 operand pairs lane class c multiplies (the
// MMA B fragment of row m).  x' = x * 2^s is the scaled copy, f = 2^-s and
// X_g the sum of x over the group, added as ((X_0 + X_1) + X_2) + X_3 from
// the sums X_c of the 32 values of each lane class c.
// The 80-byte stride keeps the 16-byte loads of 8 lanes on distinct bank
// groups.
template <int MODE> struct Pkg;
template <> struct Pkg<kMMA> { static constexpr int kRows = 8, kRowBytes = 320, kBytes = 2624; };
template <> struct Pkg<kMMA1> { static constexpr int kRows = 1, kRowBytes = 320, kBytes = 336; };
template <> struct Pkg<kMMA16> { static constexpr int kRows = 16, kRowBytes = 320, kBytes = 5248; };

// Groups per split-K segment (an item's K extent): kSegGroups (512 rows) in
// every mode, never set by the grid, so every summation order depends on the
// shape alone.  Shorter M = 1 segments (a partial is only 256 bytes there)
// speed up single small calls but cost more per-segment work on large ones.

template <int MODE>
__host__ __device__ constexpr int slot_bytes() { return kQuadTiles * kBlockBytes + Pkg<MODE>::kBytes; }
#ifndef W4G128_M1_RING_DEPTH
#define W4G128_M1_RING_DEPTH 2
#endif
// Ring slots per warp: kDepth, or for the small-package M = 1 mode
// W4G128_M1_RING_DEPTH (three 4688-byte slots per warp still fit 16 warps).
template <int MODE>
__host__ __device__ constexpr int ring_depth() { return multi_row<MODE>() ? kDepth : W4G128_M1_RING_DEPTH; }
constexpr int kMaxDepth = kDepth > W4G128_M1_RING_DEPTH ? kDepth : W4G128_M1_RING_DEPTH;
constexpr int kBarBytes = ((kNW * kMaxDepth * 8 + 127) / 128) * 128;  // per warp, its ring's mbarriers
// Warps per CTA: 16, or 8 at M <= 16: its 9.4 KB slots (a 5.1 KB package)
// leave room for fewer rings, and its twice as many accumulators need more
// than 168 registers a thread, which the register file grants only with at
// most two warps per scheduler.
template <int MODE>
__host__ __device__ constexpr int cta_warps_max() { return MODE == kMMA16 ? 8 : kNW; }
template <int MODE>
__host__ __device__ constexpr int smem_bytes() {
  return kBarBytes + cta_warps_max<MODE>() * ring_depth<MODE>() * slot_bytes<MODE>();
}

static_assert(slot_bytes<kMMA1>() % 16 == 0 && slot_bytes<kMMA>() % 16 == 0 && slot_bytes<kMMA16>() % 16 == 0,
              "bulk copies need 16-byte slots");
static_assert(Pkg<kMMA1>::kRows == 1 && Pkg<kMMA>::kRows == 8 && Pkg<kMMA16>::kRows == 16, "x rows per package");
static_assert(Pkg<kMMA1>::kBytes % 16 == 0 && Pkg<kMMA>::kBytes % 16 == 0 && Pkg<kMMA16>::kBytes % 16 == 0,
              "bulk copies need 16-byte packages");
static_assert(smem_bytes<kMMA>() <= 232448 && smem_bytes<kMMA1>() <= 232448 && smem_bytes<kMMA16>() <= 232448,
              "a CTA's rings must fit the 227 KB of shared memory");

// ----------------------------------------------------------------- parameters

struct MatParams {
  const uint8_t* packed;
  uint8_t* xpkg;        // this matrix's activation packages (in the workspace)
  const uint16_t* x;
  uint16_t* y;
  long long item_begin;  // first item of this matrix in the flat list
  int K, N;
  int quad_begin;        // first quad (and ticket) of this matrix in the flat quad list
  int g_begin;           // first (matrix, group) package index of this matrix
};

// M >= 2: warp w's split-quad record, one 64-bit word written (relaxed) at
// the start of its stream after the prep kernel has cleared it: bit 63 set
// once written; bit 62 set if the quad w's range starts in began in warp
// w - 1, so every split quad is named by exactly one record, its second
// warp's; then the quad's matrix (bits 44..52), its index in the matrix
// (bits 20..43) and the segment w starts at (bits 0..19).
constexpr unsigned long long kRecWritten = 1ull << 63, kRecSplit = 1ull << 62;
__host__ __device__ constexpr unsigned long long split_rec(bool split, int mi, int q, int s) {
  return kRecWritten | (split ? kRecSplit : 0ull) | (static_cast<unsigned long long>(mi) << 44) |
         (static_cast<unsigned long long>(q) << 20) | static_cast<unsigned long long>(s);
}
static_assert(W4G128_MAX_MATRICES <= 512, "9 bits of matrix index in a split-quad record");

// Calls of up to kFewMatrices matrices (a decoder layer's projections) use a
// kernel whose parameter block holds that many descriptors: about 0.6 KB
// instead of 28 KB to copy per launch, and the constant cache keeps all of it.
constexpr int kFewMatrices = 8;

// Local calls of up to kFewMatrices matrices take their CTAs' item ranges
// from a table the host computes; it holds up to kMaxLocalCtas CTAs.
constexpr int kMaxLocalCtas = 192;

template <int MAXMAT>
struct StreamParams {
  long long total_items;
  float* partials;       // [total_items][rows][64]: one slot per (matrix, quad, segment)
  unsigned* tickets;     // [total_quads] arrival counters of split quads (M = 1) / matrix of each quad (M >= 2)
  unsigned long long* recs;  // [W] split-quad records (M >= 2)
  unsigned* status;
  // The residual add + RMS norm call (one matrix; residual == nullptr
  // otherwise): its y is h = residual + x W, and the norm kernel writes
  // out = gamma h / rms(h).
  const uint16_t* residual;
  const uint16_t* gamma;
  uint16_t* nout;
  float eps;
  int count, M, W, total_quads, total_groups;
  int per_warp_reduce;   // M >= 2: the split quads are folded per streaming warp (else per quad)
  int red_chunk;         // M >= 2, per-quad fold: partial slots per bulk copy (8 or 16)
  int red_reverse;       // M >= 2, per-quad fold: fold CTA b takes quad total_quads - 1 - b
  int depth;             // ring slots per warp (ring_depth of the mode)
  unsigned long long wait_ns;  // limit of every device-side wait
  int cta_warps;         // warps per streaming CTA
  int local_pkg_off;     // M = 1 with CTA-local packages: shared-memory offsets of the package area
  int local_part_off;    //   and of the partial-slot area
  int pair;              // M = 1, one matrix: quad q runs on CTAs 2q and 2q + 1, a cluster of two
  // local calls of up to kFewMatrices matrices: CTA c streams items
  // [cta_begin[c], cta_begin[c + 1]), split evenly over its warps
  long long cta_begin[MAXMAT <= kFewMatrices ? kMaxLocalCtas + 1 : 1];
  MatParams mats[MAXMAT];
};

static_assert(sizeof(StreamParams<W4G128_MAX_MATRICES>) <= 32000, "kernel parameter limit");


// A matrix of the call.  With one matrix the index is the constant 0, so every
// read of its descriptor is at a fixed offset of the kernel parameters: those
// reads are independent of one another and shared by all SMs, while a
// computed index makes each a dependent lookup (an L2 round trip when it
// misses the constant cache).
template <int MAXMAT>
__device__ __forceinline__ const MatParams& mat(const StreamParams<MAXMAT>& p, int i) {
  return p.mats[MAXMAT == 1 ? 0 : i];
}

__host__ __device__ constexpr int div_up(int a, int b) { return (a + b - 1) / b; }

// ----------------------------------------------------------------- cursor

// Position of one chunk (matrix mi, quad q, segment s, group g) in the flat
// list, with the current matrix's sizes and both source pointers cached so
// that moving to the next chunk is a few increments: within a matrix the
// packed bytes are read strictly sequentially.
struct Cursor {
  long long item;
  const uint8_t* src;   // this chunk's weight blocks
  const uint8_t* xsrc;  // this chunk's activation package
  int mi, q, s, g, g_end;
  int G, S, NQ, T, ntiles;
};

template <int MODE, int MAXMAT>
__device__ __forceinline__ void cursor_load(Cursor& c, const StreamParams<MAXMAT>& p, int mi) {
  const MatParams& m = mat(p, mi);
  c.mi = mi;
  c.G = m.K / kGroup;
  c.S = div_up(c.G, kSegGroups);
  c.T = m.N / kTileN;
  c.NQ = div_up(c.T, kQuadTiles);
}

template <int MODE, int MAXMAT>
__device__ __forceinline__ void cursor_seek(Cursor& c, const StreamParams<MAXMAT>& p, long long item) {
  int lo = 0;
  if constexpr (MAXMAT > 1) {
    int hi = p.count - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.mats[mid].item_begin <= item) lo = mid; else hi = mid - 1;
    }
  }
  cursor_load<MODE>(c, p, lo);
  const long long local = item - mat(p, lo).item_begin;
  c.item = item;
  c.q = local < (1ll << 31) ? static_cast<int>(static_cast<unsigned>(local) / static_cast<unsigned>(c.S))
                            : static_cast<int>(local / c.S);
  c.s = static_cast<int>(local - static_cast<long long>(c.q) * c.S);
  c.g = c.s * kSegGroups;
  c.g_end = min(c.g + kSegGroups, c.G);
  c.ntiles = min(kQuadTiles, c.T - kQuadTiles * c.q);
  c.src = mat(p, lo).packed + static_cast<long long>(c.q) * c.G * kQuadBytes +
          static_cast<long long>(c.g) * c.ntiles * kBlockBytes;
  c.xsrc = mat(p, lo).xpkg + static_cast<long long>(c.g) * Pkg<MODE>::kBytes;
}

template <int MODE, int MAXMAT>
__device__ __forceinline__ void cursor_next(Cursor& c, const StreamParams<MAXMAT>& p) {
  c.src += c.ntiles * kBlockBytes;
  c.xsrc += Pkg<MODE>::kBytes;
  if (++c.g < c.g_end) return;
  ++c.item;
  if (++c.s < c.S) {
    c.g_end = min(c.g + kSegGroups, c.G);
    return;
  }
  c.s = 0;
  c.g = 0;
  if (++c.q < c.NQ) {  // the next quad starts where this one ended
    c.ntiles = min(kQuadTiles, c.T - kQuadTiles * c.q);
    c.xsrc = mat(p, c.mi).xpkg;
    c.g_end = min(kSegGroups, c.G);
    return;
  }
  if (c.mi + 1 == p.count) return;  // past the end; never dereferenced
  cursor_load<MODE>(c, p, c.mi + 1);
  c.q = 0;
  c.ntiles = min(kQuadTiles, c.T);
  c.src = mat(p, c.mi).packed;
  c.xsrc = mat(p, c.mi).xpkg;
  c.g_end = min(kSegGroups, c.G);
}

// What the M = 1 fold of one split quad needs, recorded by the warp that
// reaches it (32 bytes).
struct PendFold {
  long long first;  // first partial slot of the fold (the first warp's prefix fold)
  uint16_t* y;      // the quad's first output column
  int nslot;        // slots from `first` to the quad's last segment
  int cols;         // columns of the quad (64, fewer in a ragged last quad)
  int n0;           // index of the quad's first column in y
  int pad;
};

// Arrival at a split quad: returns the count before this arrival.
__device__ __forceinline__ unsigned ticket_acq_rel(unsigned* t) {
  unsigned prev;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(t) : "memory");
  return prev;
}

// floor(I w / W) for 0 <= w <= W, the first item of warp w under the
// balanced split: in 32-bit arithmetic when I W fits (any call short of
// about 1.7 million items at 2432 warps), since a 64-bit division is a
// long instruction sequence on the path to a warp's first copy.
__device__ __forceinline__ long long split_at(long long I, long long w, int W) {
  if (w >= W) return I;
  if (I * W < (1ll << 32))
    return static_cast<long long>(static_cast<unsigned>(I * w) / static_cast<unsigned>(W));
  return I * w / W;
}

// Owner warp of an item under the balanced split [floor(wI/W), floor((w+1)I/W)).
__device__ __forceinline__ int owner_of(long long item, long long I, int W) {
  const long long n = (item + 1) * W + I - 1;
  if (n < (1ll << 32) && I < (1ll << 32))
    return static_cast<int>(static_cast<unsigned>(n) / static_cast<unsigned>(I)) - 1;
  return static_cast<int>(n / I) - 1;
}

// ----------------------------------------------------------------- chunk copy

// Debug builds: the chunk's weight blocks and activation package lie inside
// their matrix's packed bytes and packages.
template <int MODE, int MAXMAT>
__device__ __forceinline__ bool chunk_in_range(const StreamParams<MAXMAT>& p, const Cursor& c) {
  if constexpr (!kDebug) {
    return true;
  } else {
    const MatParams& m = mat(p, c.mi);
    const bool w = c.src >= m.packed && c.src + c.ntiles * kBlockBytes <= m.packed + packed_bytes_of(m.K, m.N);
    const bool x = c.xsrc >= m.xpkg && c.xsrc + Pkg<MODE>::kBytes <= m.xpkg + static_cast<long long>(m.K / kGroup) *
                                                                                 Pkg<MODE>::kBytes;
    return dbg_ok(p.status, w && x);
  }
}

// The chunk (quad q, group g) is nt(q) adjacent blocks: one bulk copy.
// Debug builds skip a copy outside its buffers (an arrival completes the
// slot instead).
template <int MODE, int MAXMAT>
__device__ __forceinline__ void issue_weights(const StreamParams<MAXMAT>& p, const Cursor& c, uint32_t slot,
                                              uint32_t bar, uint64_t pol) {
  if (!chunk_in_range<MODE>(p, c)) {
    mbar_arrive_plain(bar);
    return;
  }
  mbar_arrive_expect_tx(bar, c.ntiles * kBlockBytes + Pkg<MODE>::kBytes);
  bulk_g2s(slot, c.src, c.ntiles * kBlockBytes, bar, pol);
}

template <int MODE, int MAXMAT>
__device__ __forceinline__ void issue_package(const StreamParams<MAXMAT>& p, const Cursor& c, uint32_t slot,
                                              uint32_t bar, uint64_t pol) {
  if constexpr (kDebug) {
    const MatParams& m = mat(p, c.mi);
    const bool w = c.src >= m.packed && c.src + c.ntiles * kBlockBytes <= m.packed + packed_bytes_of(m.K, m.N);
    const bool x = c.xsrc >= m.xpkg && c.xsrc + Pkg<MODE>::kBytes <= m.xpkg + static_cast<long long>(m.K / kGroup) *
                                                                                 Pkg<MODE>::kBytes;
    if (!(w && x)) return;  // recorded (and the slot completed) by issue_weights
  }
  bulk_g2s(slot + kQuadTiles * kBlockBytes, c.xsrc, Pkg<MODE>::kBytes, bar, pol);
}

// ----------------------------------------------------------------- in-register dequantisation

// Word layout (per lane r = l/4, c = l%4): nibble p = 4b + 2a + e holds row
// 2c + 8a + b of column r + 8e.  With v = w >> 8, LOP3 with the fp16 magic
// 0x6400 (1024) turns
//   w & 0x000F000F -> nibbles 0, 4 (rows 2c, 2c+1, column r)      as 1024 + q
//   w & 0x00F000F0 -> nibbles 1, 5 (rows 2c, 2c+1, column r+8)    as 1024 + 16q
//   v & 0x000F000F -> nibbles 2, 6 (rows 2c+8, 2c+9, column r)    as 1024 + q
//   v & 0x00F000F0 -> nibbles 3, 7 (rows 2c+8, 2c+9, column r+8)  as 1024 + 16q
// into fp16 pairs, which are the A fragment of the warp MMA below.
constexpr uint32_t kMagic = 0x64006400u;  // fp16 1024.0 in both halves

// Warp MMA: D[16 cols x 8 rows] += A[16 cols x 16 k] * B[16 k x 8 rows]; the
// four LOP3 outputs of one packed word are exactly this lane's A fragment
// (columns r + 8 carry 1024 + 16q, so their D rows are scaled accordingly).
__device__ __forceinline__ void mma_word(uint32_t w, uint32_t xa, uint32_t xb, float (&d)[4]) {
  const uint32_t v = w >> 8;
  const uint32_t a0 = lop3_and_or(w, 0x000F000Fu, kMagic);
  const uint32_t a1 = lop3_and_or(w, 0x00F000F0u, kMagic);
  const uint32_t a2 = lop3_and_or(v, 0x000F000Fu, kMagic);
  const uint32_t a3 = lop3_and_or(v, 0x00F000F0u, kMagic);
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(xa), "r"(xb));
}

// The same A fragment against two 8-row x tiles (rows 0-7 into d, 8-15 into e):
// each is exactly the MMA mma_word issues for its rows.
__device__ __forceinline__ void mma_word2(uint32_t w, uint32_t xa, uint32_t xb, uint32_t ya, uint32_t yb,
                                          float (&d)[4], float (&e)[4]) {
  const uint32_t v = w >> 8;
  const uint32_t a0 = lop3_and_or(w, 0x000F000Fu, kMagic);
  const uint32_t a1 = lop3_and_or(w, 0x00F000F0u, kMagic);
  const uint32_t a2 = lop3_and_or(v, 0x000F000Fu, kMagic);
  const uint32_t a3 = lop3_and_or(v, 0x00F000F0u, kMagic);
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(xa), "r"(xb));
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(e[0]), "+f"(e[1]), "+f"(e[2]), "+f"(e[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(ya), "r"(yb));
}

// Two IEEE fp32 FMAs in one instruction (Blackwell packed f32x2); each lane of
// the pair rounds exactly like fmaf.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 A, B, C;\n\t"
      "mov.b64 A, {%2, %3};\n\t"
      "mov.b64 B, {%4, %5};\n\t"
      "mov.b64 C, {%6, %7};\n\t"
      "fma.rn.f32x2 C, A, B, C;\n\t"
      "mov.b64 {%0, %1}, C;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 A, B;\n\t"
      "mov.b64 A, {%2, %3};\n\t"
      "mov.b64 B, {%4, %5};\n\t"
      "mul.rn.f32x2 A, A, B;\n\t"
      "mov.b64 {%0, %1}, A;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint16_t to_bf16(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

// Output element i of a matrix from its fp32 sum v: bf16(v), or, in the
// residual add + RMS norm call, h = bf16(residual + v) -- one rounding, the
// add kept apart from any multiply.  The element's residual is read by the
// thread that writes it, so h may overwrite the residual in place.
template <bool NORM, int MAXMAT>
__device__ __forceinline__ uint16_t emit(const StreamParams<MAXMAT>& p, long long i, float v) {
  if constexpr (NORM) v = __fadd_rn(v, __uint_as_float(static_cast<uint32_t>(__ldcg(p.residual + i)) << 16));
  return to_bf16(v);
}

// The residual's elements i, i + 1 (i even) as one 32-bit word (0 without
// the norm); loaded ahead of the sums it is added to.
template <bool NORM, int MAXMAT>
__device__ __forceinline__ uint32_t residual2(const StreamParams<MAXMAT>& p, long long i) {
  if constexpr (NORM) return __ldcg(reinterpret_cast<const uint32_t*>(p.residual + i));
  else return 0u;
}

// Elements i, i + 1 as one 32-bit word, given residual2 of them.
template <bool NORM>
__device__ __forceinline__ uint32_t emit2(float a, float b, uint32_t r) {
  if constexpr (NORM) {
    a = __fadd_rn(a, bf16_lo(r));
    b = __fadd_rn(b, bf16_hi(r));
  }
  return static_cast<uint32_t>(to_bf16(a)) | (static_cast<uint32_t>(to_bf16(b)) << 16);
}

// Rows of the per-lane accumulators: the MMA keeps (r, 2c), (r, 2c+1),
// (r+8, 2c), (r+8, 2c+1) (and the same for rows 8 + 2c, 9 + 2c at M > 8);
// M = 1 keeps (column r, column r+8) of x row 2c, which every lane class
// holds alike.
template <int MODE> struct Acc {
  static constexpr int kN = (MODE == kMMA1) ? 2 : (MODE == kMMA16 ? 8 : 4);
};

// One chunk: every tile of the quad for one group (weights in the ring slot
// sl, the group's activation package at pk), added into seg[t][*].
// ILP: 0 -- tile by tile; 1 -- a whole quad's tiles in pairs, both tiles'
// MMAs interleaved; 2 (M <= 8) -- all four tiles interleaved.  Each
// accumulator receives the same MMAs in the same order in every form: the
// same bits; the interleaved forms hold more registers and keep a warp that
// is alone on its scheduler from waiting on one tile's dependent chain.
template <int MODE, int ILP = 0>
__device__ __forceinline__ void compute_chunk(const uint8_t* sl, const uint8_t* pk, int ntiles, int lane,
                                              float (&seg)[kQuadTiles][Acc<MODE>::kN]) {
  const int r = lane >> 2, c = lane & 3;
  const int row = multi_row<MODE>() ? r : 0;
  const uint32_t* xr = reinterpret_cast<const uint32_t*>(pk + row * Pkg<MODE>::kRowBytes + c * 80);
  uint32_t xw[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = reinterpret_cast<const uint4*>(xr)[i];
    xw[4 * i] = v.x; xw[4 * i + 1] = v.y; xw[4 * i + 2] = v.z; xw[4 * i + 3] = v.w;
  }
  if constexpr (MODE == kMMA16) {
    // rows r (tile 0) and 8 + r (tile 1) of the B operand; (X_g, f) of rows
    // 2c, 2c + 1 and 8 + 2c, 9 + 2c.  Each tile goes through exactly the
    // arithmetic of the 8-row mode, so every row's bits match it.
    const uint32_t* yr = reinterpret_cast<const uint32_t*>(pk + (8 + r) * Pkg<MODE>::kRowBytes + c * 80);
    uint32_t yw[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = reinterpret_cast<const uint4*>(yr)[i];
      yw[4 * i] = v.x; yw[4 * i + 1] = v.y; yw[4 * i + 2] = v.z; yw[4 * i + 3] = v.w;
    }
    const float* tl = reinterpret_cast<const float*>(pk + Pkg<MODE>::kRows * Pkg<MODE>::kRowBytes);
    const float4 xq0 = *reinterpret_cast<const float4*>(tl + 4 * c);
    const float4 xq1 = *reinterpret_cast<const float4*>(tl + 16 + 4 * c);
    // tile t's scale/min epilogue of one 8-row half (accumulator chains a, b)
    auto epilogue = [&](uint2 me, const float (&a)[4], const float (&b)[4], const float4 xq, float& s0, float& s1,
                        float& s2, float& s3) {
      const float sl0 = bf16_lo(me.x), sh0 = bf16_lo(me.y);
      const float ml0 = fmaf(-1024.f, sl0, bf16_hi(me.x));
      const float mh0 = fmaf(-64.f, sh0, bf16_hi(me.y));
      const float2 Xab = make_float2(xq.x, xq.z);
      const float2 fab = make_float2(xq.y, xq.w);
      const float2 fab16 = make_float2(xq.y * 0.0625f, xq.w * 0.0625f);
      float2 lo2 = ffma2(make_float2(ml0, ml0), Xab, make_float2(s0, s1));
      lo2 = ffma2(fmul2(make_float2(sl0, sl0), fab), make_float2(a[0] + b[0], a[1] + b[1]), lo2);
      float2 hi2 = ffma2(make_float2(mh0, mh0), Xab, make_float2(s2, s3));
      hi2 = ffma2(fmul2(make_float2(sh0, sh0), fab16), make_float2(a[2] + b[2], a[3] + b[3]), hi2);
      s0 = lo2.x;
      s1 = lo2.y;
      s2 = hi2.x;
      s3 = hi2.y;
    };
    if (ILP > 0 && ntiles == kQuadTiles) {
      // A whole quad, tiles in pairs with their MMAs interleaved; every
      // accumulator receives the same MMAs in the same order as below.
#pragma unroll
      for (int t = 0; t < kQuadTiles; t += 2) {
        const uint8_t* blk = sl + t * kBlockBytes;
        const uint4 a0 = *reinterpret_cast<const uint4*>(blk + 16 * lane);
        const uint4 a1 = *reinterpret_cast<const uint4*>(blk + 512 + 16 * lane);
        const uint2 ma = *reinterpret_cast<const uint2*>(blk + kCodeBytes + 8 * r);
        const uint4 b0 = *reinterpret_cast<const uint4*>(blk + kBlockBytes + 16 * lane);
        const uint4 b1 = *reinterpret_cast<const uint4*>(blk + kBlockBytes + 512 + 16 * lane);
        const uint2 mb = *reinterpret_cast<const uint2*>(blk + kBlockBytes + kCodeBytes + 8 * r);
        float da0[4] = {0.f, 0.f, 0.f, 0.f}, da1[4] = {0.f, 0.f, 0.f, 0.f};
        float ea0[4] = {0.f, 0.f, 0.f, 0.f}, ea1[4] = {0.f, 0.f, 0.f, 0.f};
        float db0[4] = {0.f, 0.f, 0.f, 0.f}, db1[4] = {0.f, 0.f, 0.f, 0.f};
        float eb0[4] = {0.f, 0.f, 0.f, 0.f}, eb1[4] = {0.f, 0.f, 0.f, 0.f};
        mma_word2(a0.x, xw[0], xw[1], yw[0], yw[1], da0, ea0);
        mma_word2(b0.x, xw[0], xw[1], yw[0], yw[1], db0, eb0);
        mma_word2(a0.y, xw[2], xw[3], yw[2], yw[3], da1, ea1);
        mma_word2(b0.y, xw[2], xw[3], yw[2], yw[3], db1, eb1);
        mma_word2(a0.z, xw[4], xw[5], yw[4], yw[5], da0, ea0);
        mma_word2(b0.z, xw[4], xw[5], yw[4], yw[5], db0, eb0);
        mma_word2(a0.w, xw[6], xw[7], yw[6], yw[7], da1, ea1);
        mma_word2(b0.w, xw[6], xw[7], yw[6], yw[7], db1, eb1);
        mma_word2(a1.x, xw[8], xw[9], yw[8], yw[9], da0, ea0);
        mma_word2(b1.x, xw[8], xw[9], yw[8], yw[9], db0, eb0);
        mma_word2(a1.y, xw[10], xw[11], yw[10], yw[11], da1, ea1);
        mma_word2(b1.y, xw[10], xw[11], yw[10], yw[11], db1, eb1);
        mma_word2(a1.z, xw[12], xw[13], yw[12], yw[13], da0, ea0);
        mma_word2(b1.z, xw[12], xw[13], yw[12], yw[13], db0, eb0);
        mma_word2(a1.w, xw[14], xw[15], yw[14], yw[15], da1, ea1);
        mma_word2(b1.w, xw[14], xw[15], yw[14], yw[15], db1, eb1);
        epilogue(ma, da0, da1, xq0, seg[t][0], seg[t][1], seg[t][2], seg[t][3]);
        epilogue(ma, ea0, ea1, xq1, seg[t][4], seg[t][5], seg[t][6], seg[t][7]);
        epilogue(mb, db0, db1, xq0, seg[t + 1][0], seg[t + 1][1], seg[t + 1][2], seg[t + 1][3]);
        epilogue(mb, eb0, eb1, xq1, seg[t + 1][4], seg[t + 1][5], seg[t + 1][6], seg[t + 1][7]);
      }
      return;
    }
#pragma unroll
    for (int t = 0; t < kQuadTiles; ++t) {
      if (t < ntiles) {
        const uint8_t* blk = sl + t * kBlockBytes;
        const uint4 u0 = *reinterpret_cast<const uint4*>(blk + 16 * lane);
        const uint4 u1 = *reinterpret_cast<const uint4*>(blk + 512 + 16 * lane);
        const uint2 me = *reinterpret_cast<const uint2*>(blk + kCodeBytes + 8 * r);
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
        float e0[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
        mma_word2(u0.x, xw[0], xw[1], yw[0], yw[1], d0, e0);
        mma_word2(u0.y, xw[2], xw[3], yw[2], yw[3], d1, e1);
        mma_word2(u0.z, xw[4], xw[5], yw[4], yw[5], d0, e0);
        mma_word2(u0.w, xw[6], xw[7], yw[6], yw[7], d1, e1);
        mma_word2(u1.x, xw[8], xw[9], yw[8], yw[9], d0, e0);
        mma_word2(u1.y, xw[10], xw[11], yw[10], yw[11], d1, e1);
        mma_word2(u1.z, xw[12], xw[13], yw[12], yw[13], d0, e0);
        mma_word2(u1.w, xw[14], xw[15], yw[14], yw[15], d1, e1);
        epilogue(me, d0, d1, xq0, seg[t][0], seg[t][1], seg[t][2], seg[t][3]);
        epilogue(me, e0, e1, xq1, seg[t][4], seg[t][5], seg[t][6], seg[t][7]);
      }
    }
  } else {
    // (X_g, f) of rows 2c and 2c + 1; with one x row (kMMA1) every lane takes
    // row 0's pair, and only lanes c == 0 (row 0) are ever stored
    float4 xq;
    if constexpr (MODE == kMMA) {
      xq = *reinterpret_cast<const float4*>(pk + Pkg<MODE>::kRows * Pkg<MODE>::kRowBytes + 16 * c);
    } else {
      const float2 t0 = *reinterpret_cast<const float2*>(pk + Pkg<MODE>::kRowBytes);
      xq = make_float4(t0.x, t0.y, t0.x, t0.y);
    }
    const float2 Xab = make_float2(xq.x, xq.z);
    const float2 fab = make_float2(xq.y, xq.w);
    const float2 fab16 = make_float2(xq.y * 0.0625f, xq.w * 0.0625f);
    // Tile t's sums: (1024 + q) x' (columns r) and (1024 + 16q) x' (columns
    // r + 8) as (column, row) fragments in two chains, words 0, 2, 4, 6 into
    // d0 and 1, 3, 5, 7 into d1; then its scale/min epilogue into seg[t].
    auto epilogue = [&](int t, uint2 me, const float (&d0)[4], const float (&d1)[4]) {
      const float sl0 = bf16_lo(me.x), sh0 = bf16_lo(me.y);
      const float ml0 = fmaf(-1024.f, sl0, bf16_hi(me.x));
      const float mh0 = fmaf(-64.f, sh0, bf16_hi(me.y));
      if constexpr (MODE == kMMA1) {
        // the first lane of each pair below, alone: the same roundings
        seg[t][0] = __fmaf_rn(__fmul_rn(sl0, fab.x), d0[0] + d1[0], __fmaf_rn(ml0, Xab.x, seg[t][0]));
        seg[t][1] = __fmaf_rn(__fmul_rn(sh0, fab16.x), d0[2] + d1[2], __fmaf_rn(mh0, Xab.x, seg[t][1]));
      } else {
        float2 lo2 = ffma2(make_float2(ml0, ml0), Xab, make_float2(seg[t][0], seg[t][1]));
        lo2 = ffma2(fmul2(make_float2(sl0, sl0), fab), make_float2(d0[0] + d1[0], d0[1] + d1[1]), lo2);
        float2 hi2 = ffma2(make_float2(mh0, mh0), Xab, make_float2(seg[t][2], seg[t][3]));
        hi2 = ffma2(fmul2(make_float2(sh0, sh0), fab16), make_float2(d0[2] + d1[2], d0[3] + d1[3]), hi2);
        seg[t][0] = lo2.x;
        seg[t][1] = lo2.y;
        seg[t][2] = hi2.x;
        seg[t][3] = hi2.y;
      }
    };
    if (ILP == 2 && ntiles == kQuadTiles) {
      uint4 u0[kQuadTiles], u1[kQuadTiles];
      uint2 me[kQuadTiles];
#pragma unroll
      for (int t = 0; t < kQuadTiles; ++t) {
        const uint8_t* blk = sl + t * kBlockBytes;
        u0[t] = *reinterpret_cast<const uint4*>(blk + 16 * lane);
        u1[t] = *reinterpret_cast<const uint4*>(blk + 512 + 16 * lane);
        me[t] = *reinterpret_cast<const uint2*>(blk + kCodeBytes + 8 * r);
      }
      float d0[kQuadTiles][4], d1[kQuadTiles][4];
#pragma unroll
      for (int t = 0; t < kQuadTiles; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) d0[t][e] = d1[t][e] = 0.f;
#pragma unroll
      for (int t = 0; t < kQuadTiles; ++t) mma_word(u0[t].x, xw[0], xw[1], d0[t]);
#pragma unroll
      for (int t = 0; t < kQuadTiles; ++t) mma_word(u0[t].y, xw[2], xw[3], d1[t]);
#pragma unroll
      for (int t = 0; t < kQuadTiles; ++t) mma_word(u0[t].z, xw[4], xw[5], d0[t]);
#pragma unroll
      for (int t = 0; t < kQuadTiles; ++t) mma_word(u0[t].w, xw[6], xw[7], d1[t]);
#pragma unroll
      for (int t = 0; t < kQuadTiles; ++t) mma_word(u1[t].x, xw[8], xw[9], d0[t]);
#pragma unroll
      for (int t = 0; t < kQuadTiles; ++t) mma_word(u1[t].y, xw[10], xw[11], d1[t]);
#pragma unroll
      for (int t = 0; t < kQuadTiles; ++t) mma_word(u1[t].z, xw[12], xw[13], d0[t]);
#pragma unroll
      for (int t = 0; t < kQuadTiles; ++t) mma_word(u1[t].w, xw[14], xw[15], d1[t]);
#pragma unroll
      for (int t = 0; t < kQuadTiles; ++t) epilogue(t, me[t], d0[t], d1[t]);
      return;
    }
    if (ILP == 1 && ntiles == kQuadTiles) {
#pragma unroll
      for (int t = 0; t < kQuadTiles; t += 2) {
        const uint8_t* blk = sl + t * kBlockBytes;
        const uint4 a0 = *reinterpret_cast<const uint4*>(blk + 16 * lane);
        const uint4 a1 = *reinterpret_cast<const uint4*>(blk + 512 + 16 * lane);
        const uint2 ma = *reinterpret_cast<const uint2*>(blk + kCodeBytes + 8 * r);
        const uint4 b0 = *reinterpret_cast<const uint4*>(blk + kBlockBytes + 16 * lane);
        const uint4 b1 = *reinterpret_cast<const uint4*>(blk + kBlockBytes + 512 + 16 * lane);
        const uint2 mb = *reinterpret_cast<const uint2*>(blk + kBlockBytes + kCodeBytes + 8 * r);
        float da0[4] = {0.f, 0.f, 0.f, 0.f}, da1[4] = {0.f, 0.f, 0.f, 0.f};
        float db0[4] = {0.f, 0.f, 0.f, 0.f}, db1[4] = {0.f, 0.f, 0.f, 0.f};
        mma_word(a0.x, xw[0], xw[1], da0);
        mma_word(b0.x, xw[0], xw[1], db0);
        mma_word(a0.y, xw[2], xw[3], da1);
        mma_word(b0.y, xw[2], xw[3], db1);
        mma_word(a0.z, xw[4], xw[5], da0);
        mma_word(b0.z, xw[4], xw[5], db0);
        mma_word(a0.w, xw[6], xw[7], da1);
        mma_word(b0.w, xw[6], xw[7], db1);
        mma_word(a1.x, xw[8], xw[9], da0);
        mma_word(b1.x, xw[8], xw[9], db0);
        mma_word(a1.y, xw[10], xw[11], da1);
        mma_word(b1.y, xw[10], xw[11], db1);
        mma_word(a1.z, xw[12], xw[13], da0);
        mma_word(b1.z, xw[12], xw[13], db0);
        mma_word(a1.w, xw[14], xw[15], da1);
        mma_word(b1.w, xw[14], xw[15], db1);
        epilogue(t, ma, da0, da1);
        epilogue(t + 1, mb, db0, db1);
      }
      return;
    }
#pragma unroll
    for (int t = 0; t < kQuadTiles; ++t) {
      if (t < ntiles) {
        const uint8_t* blk = sl + t * kBlockBytes;
        const uint4 u0 = *reinterpret_cast<const uint4*>(blk + 16 * lane);
        const uint4 u1 = *reinterpret_cast<const uint4*>(blk + 512 + 16 * lane);
        const uint2 me = *reinterpret_cast<const uint2*>(blk + kCodeBytes + 8 * r);
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
        mma_word(u0.x, xw[0], xw[1], d0);
        mma_word(u0.y, xw[2], xw[3], d1);
        mma_word(u0.z, xw[4], xw[5], d0);
        mma_word(u0.w, xw[6], xw[7], d1);
        mma_word(u1.x, xw[8], xw[9], d0);
        mma_word(u1.y, xw[10], xw[11], d1);
        mma_word(u1.z, xw[12], xw[13], d0);
        mma_word(u1.w, xw[14], xw[15], d1);
        epilogue(t, me, d0, d1);
      }
    }
  }
}

// ----------------------------------------------------------------- the streaming kernel

// CTAs of at most kWideWarps warps (calls too small to give every SM 16
// warps) run forms of the streaming kernels with 168 registers, which
// interleave all four tiles of a quad: there a warp is often alone on its
// scheduler.
constexpr int kWideWarps = 12;

template <int MODE, int MAXMAT, bool NORM, bool WIDE = false>
// M = 1 is held to 120 registers (no spills): 4096 of the
// SM's 65536 registers stay free for the next call's one-warp prep CTAs.
// M <= 16 (8 warps) may use up to 255; the WIDE form of M <= 8 168.
__global__ void __launch_bounds__((WIDE ? kWideWarps : cta_warps_max<MODE>()) * 32, 1)
    __maxnreg__(WIDE ? 168 : (MODE == kMMA1 ? 120 : (MODE == kMMA16 ? 255 : 128)))
    stream_kernel(const __grid_constant__ StreamParams<MAXMAT> p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int NA = Acc<MODE>::kN;
  constexpr int kSlot = slot_bytes<MODE>();
  // Ring slots per warp, read from the parameters although fixed per mode:
  // with a compile-time depth the compiler schedules the MMA modes' main loop
  // worse (measured: layer step M = 8 44.2 vs 43.0 us, lm_head M = 8 113.2 vs
  // 109.9 us).
  const int D = p.depth;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, c = lane & 3;
  const int wg = blockIdx.x * (blockDim.x >> 5) + warp;  // CTAs hold up to kNW warps
  // M = 1: split quads whose last ticket a warp of this CTA took; folded by
  // the whole CTA after its stream (the only block-wide barriers are here and
  // before that fold).  Each warp records what the fold of its (at most two)
  // split quads needs when it reaches them, so the fold after the barrier
  // reads only shared memory (no lookups in the matrix table, no divisions).
  __shared__ int fold_n;
  __shared__ int fold_ref[2 * kNW];     // entries of pend_info to fold
  __shared__ PendFold pend_info[2 * kNW];
  if constexpr (!multi_row<MODE>()) {
    if (threadIdx.x == 0) fold_n = 0;
    __syncthreads();
  }

  const long long I = p.total_items;
  const long long it_a = split_at(I, wg, p.W), it_b = split_at(I, wg + 1, p.W);
  // A warp's contiguous range holds at most two split quads (its first and its
  // last); their tickets are taken after the stream, so no ticket stalls it.
  int pend_q0 = 0, pend_q1 = 0;  // global quad indices
  unsigned pend_e0 = 0u, pend_e1 = 0u;  // warps contributing to each
  int n_pend = 0;
  bool failed = false;
  if (wg < p.W) {

    const uint32_t bar0 = smem_addr(smem) + warp * D * 8;
    const uint32_t ring0 = smem_addr(smem) + kBarBytes + warp * D * kSlot;
    const uint8_t* ring = smem + kBarBytes + warp * D * kSlot;

    uint64_t pol_w = 0, pol_x = 0;
    if (lane == 0) {
      for (int d = 0; d < D; ++d) mbar_init(bar0 + 8 * d, 1);
      fence_mbar_init();
      pol_w = l2_policy_evict_first();
      pol_x = l2_policy_evict_last();
    }
    __syncwarp();

    Cursor cc, ic;  // compute cursor, issue cursor
    cursor_seek<MODE>(cc, p, it_a);
    ic = cc;
    // Prologue: the weight bytes do not depend on the prep kernel, so start them
    // before waiting for it; the activation packages follow after the wait.
    // Every lane walks the cursors; lane 0 alone issues copies.  One chunk
    // starts early: the streaming CTAs become resident while the previous
    // call's kernels finish, and a deeper early prefetch competes with that
    // call's tail and with the prep kernel (measured on back-to-back layer
    // steps at M = 1: 40.4 -> 40.1 us; lm_head M = 8 115.1 -> 113.8 us).
    constexpr int kEarly = 1;
    Cursor pre[kEarly];
    int n_pre = 0;
#pragma unroll
    for (int d = 0; d < kEarly; ++d) {
      if (ic.item < it_b) {
        if (lane == 0) issue_weights<MODE>(p, ic, ring0 + d * kSlot, bar0 + 8 * d, pol_w);
        pre[d] = ic;
        ++n_pre;
        cursor_next<MODE>(ic, p);
      }
    }
    grid_dependency_wait();
    if (lane == 0) {
#pragma unroll
      for (int d = 0; d < kEarly; ++d)
        if (d < n_pre) issue_package<MODE>(p, pre[d], ring0 + d * kSlot, bar0 + 8 * d, pol_x);
    }
    unsigned issued = static_cast<unsigned>(n_pre);
    while (issued < static_cast<unsigned>(D) && ic.item < it_b) {  // the rest of the ring
      if (lane == 0) {
        issue_weights<MODE>(p, ic, ring0 + issued * kSlot, bar0 + 8 * issued, pol_w);
        issue_package<MODE>(p, ic, ring0 + issued * kSlot, bar0 + 8 * issued, pol_x);
      }
      cursor_next<MODE>(ic, p);
      ++issued;
    }
    // M >= 2: the reduce kernel may start launching now; it waits for this
    // grid to finish before it reads any partial.
    grid_dependents_launch();
    if (multi_row<MODE>() && MAXMAT > 1 && p.per_warp_reduce && lane == 0) {
      // this warp's split-quad record (the prep kernel has cleared it): does
      // the quad its range starts in begin in warp wg - 1?
      const bool split = cc.s != 0 && it_a - cc.s >= I * (wg - 1) / p.W;
      st_relaxed_u64(p.recs + wg, split_rec(split, cc.mi, cc.q, cc.s));
    }

    float seg[kQuadTiles][NA];
    float tot[kQuadTiles][NA];
#pragma unroll
    for (int t = 0; t < kQuadTiles; ++t)
#pragma unroll
      for (int e = 0; e < NA; ++e) seg[t][e] = tot[t][e] = 0.f;

    unsigned done = 0;  // chunks consumed
    int slot = 0;          // done % D
    uint32_t parity = 0u;  // (done / D) & 1
    while (cc.item < it_b) {
      if (!mbar_wait_bounded(bar0 + 8 * slot, parity, p.wait_ns)) {
        // Give up: record the timeout, drain this warp's copies in flight
        // (again bounded) and leave.  Quads this warp shared stay unreduced.
        if (lane == 0) {
          atomicCAS(p.status, 0u, static_cast<unsigned>(W4G128_ERR_TIMEOUT));
          for (unsigned k = done + 1; k < issued; ++k)
            (void)mbar_wait_bounded(bar0 + 8 * static_cast<int>(k % D), (k / D) & 1u, p.wait_ns);
        }
        __syncwarp();
        failed = true;
        break;
      }
      const int ntiles = cc.ntiles;
      const uint8_t* sl = ring + slot * kSlot;
      compute_chunk<MODE, MODE == kMMA1 ? 0 : (WIDE ? 2 : 1)>(sl, sl + kQuadTiles * kBlockBytes, ntiles, lane, seg);

      // Slot consumed: refill it with the chunk D ahead.
      __syncwarp();
      if (ic.item < it_b) {
        if (lane == 0) {
          fence_proxy_async_smem();
          const uint32_t sa = ring0 + slot * kSlot, ba = bar0 + 8 * slot;
          issue_weights<MODE>(p, ic, sa, ba, pol_w);
          issue_package<MODE>(p, ic, sa, ba, pol_x);
        }
        cursor_next<MODE>(ic, p);
        ++issued;
      }
      ++done;
      if (++slot == D) {
        slot = 0;
        parity ^= 1u;
      }

      if (cc.g + 1 == cc.g_end) {
        // ---- end of a segment
        const MatParams& m = mat(p, cc.mi);
        const int S = cc.S;
        const long long q_first = m.item_begin + static_cast<long long>(cc.q) * S;
        const long long q_last = q_first + S - 1;
        const bool owned = (q_first >= it_a) && (q_last < it_b);
        // A run holding the quad's first segments but not all of them (the
        // quad continues in later warps) keeps their left fold too and stores it
        // as one partial: the fold over segments then starts from it.
        const bool prefix = (q_first >= it_a) && !owned;
        const int rows = multi_row<MODE>() ? p.M : 1;
        if (owned || prefix) {
#pragma unroll
          for (int t = 0; t < kQuadTiles; ++t)
#pragma unroll
            for (int e = 0; e < NA; ++e) tot[t][e] = (cc.s == 0) ? seg[t][e] : tot[t][e] + seg[t][e];
        }
        if (!owned && (!prefix || cc.item + 1 == it_b) && dbg_ok(p.status, cc.item < I)) {
          // one slot per (matrix, quad, segment): the segment sum, or at the last
          // segment of a prefix run the fold of segments 0 .. s
          float* part = p.partials + cc.item * rows * 64;
          if constexpr (MODE == kMMA1) {
            // lanes c == 0 store columns r and r + 8 of every tile
            if (c == 0) {
#pragma unroll
              for (int t = 0; t < kQuadTiles; ++t) {
                if (t < ntiles) {
                  part[16 * t + r] = prefix ? tot[t][0] : seg[t][0];
                  part[16 * t + r + 8] = prefix ? tot[t][1] : seg[t][1];
                }
              }
            }
          } else {
            // accumulator 4h + {0, 1, 2, 3}: rows 8h + 2c, 8h + 2c + 1 of columns r, r + 8
#pragma unroll
            for (int t = 0; t < kQuadTiles; ++t) {
              if (t < ntiles) {
#pragma unroll
                for (int h = 0; h < NA / 4; ++h) {
                  const int r0 = 8 * h + 2 * c;
                  if (r0 < rows) {
                    part[r0 * 64 + 16 * t + r] = prefix ? tot[t][4 * h] : seg[t][4 * h];
                    part[r0 * 64 + 16 * t + r + 8] = prefix ? tot[t][4 * h + 2] : seg[t][4 * h + 2];
                  }
                  if (r0 + 1 < rows) {
                    part[(r0 + 1) * 64 + 16 * t + r] = prefix ? tot[t][4 * h + 1] : seg[t][4 * h + 1];
                    part[(r0 + 1) * 64 + 16 * t + r + 8] = prefix ? tot[t][4 * h + 3] : seg[t][4 * h + 3];
                  }
                }
              }
            }
          }
        }
#pragma unroll
        for (int t = 0; t < kQuadTiles; ++t)
#pragma unroll
          for (int e = 0; e < NA; ++e) seg[t][e] = 0.f;

        const bool quad_end = (cc.s == S - 1) || (cc.item + 1 == it_b);
        if (quad_end) {
          const int n0 = kQuadTiles * kTileN * cc.q;
          if (owned && dbg_ok(p.status, n0 + kTileN * ntiles <= m.N)) {
            if constexpr (MODE == kMMA1) {
              if (c == 0) {
#pragma unroll
                for (int t = 0; t < kQuadTiles; ++t) {
                  if (t < ntiles) {
                    const int n = n0 + 16 * t + r;
                    m.y[n] = emit<NORM>(p, n, tot[t][0]);
                    m.y[n + 8] = emit<NORM>(p, n + 8, tot[t][1]);
                  }
                }
              }
            } else {
#pragma unroll
              for (int t = 0; t < kQuadTiles; ++t) {
                if (t < ntiles) {
                  const int n = n0 + 16 * t + r;
#pragma unroll
                  for (int h = 0; h < NA / 4; ++h) {
                    const int r0 = 8 * h + 2 * c;
                    if (r0 < rows) {
                      const long long i = static_cast<long long>(r0) * m.N + n;
                      m.y[i] = emit<NORM>(p, i, tot[t][4 * h]);
                      m.y[i + 8] = emit<NORM>(p, i + 8, tot[t][4 * h + 2]);
                    }
                    if (r0 + 1 < rows) {
                      const long long i = static_cast<long long>(r0 + 1) * m.N + n;
                      m.y[i] = emit<NORM>(p, i, tot[t][4 * h + 1]);
                      m.y[i + 8] = emit<NORM>(p, i + 8, tot[t][4 * h + 3]);
                    }
                  }
                }
              }
            }
          } else if (!multi_row<MODE>() && n_pend < 2) {
            // Split quad at M = 1: its partials are written; the ticket comes after
            // the stream.  (M >= 2: the reduce kernel folds every split quad.)
            const int gq = m.quad_begin + cc.q;
            const int w_first = owner_of(q_first, I, p.W);
            const unsigned e = static_cast<unsigned>(owner_of(q_last, I, p.W) - w_first + 1);
            if (lane == 0) {
              // the fold reads the quad's slots from its first warp's prefix fold on
              const long long first = I * (w_first + 1) / p.W - 1;
              PendFold& f = pend_info[2 * warp + n_pend];
              f.first = first;
              f.y = m.y + n0;
              f.nslot = static_cast<int>(q_last + 1 - first);
              f.cols = kTileN * ntiles;
              f.n0 = n0;
            }
            if (n_pend == 0) {
              pend_q0 = gq;
              pend_e0 = e;
            } else {
              pend_q1 = gq;
              pend_e1 = e;
            }
            ++n_pend;
          }
        }
      }
      cursor_next<MODE>(cc, p);
    }
    if (!failed && n_pend > 0) {
      // The tickets are acq_rel atomics: the release publishes this warp's
      // partials (the other lanes' stores are ordered before it by the warp
      // barrier), and the acquire of the quad's last ticket makes every other
      // contributor's partials visible to this CTA (its threads are ordered
      // after it by the barrier before the fold).  No full fence is needed.
      __syncwarp();
      if (lane == 0 && dbg_ok(p.status, pend_q0 < p.total_quads && (n_pend < 2 || pend_q1 < p.total_quads))) {
        // the warp holding a quad's last ticket hands the quad to its CTA's fold
        if (ticket_acq_rel(p.tickets + pend_q0) + 1 == pend_e0) fold_ref[atomicAdd(&fold_n, 1)] = 2 * warp;
        if (n_pend > 1 && ticket_acq_rel(p.tickets + pend_q1) + 1 == pend_e1)
          fold_ref[atomicAdd(&fold_n, 1)] = 2 * warp + 1;
      }
      __syncwarp();
    }
  }  // warp in range
  if constexpr (multi_row<MODE>()) return;  // M >= 2: the reduce kernel folds
  __syncthreads();  // orders the fold after the acquiring tickets of this CTA's warps

  // ---- fold the completed split quads: one thread per (quad, 4 columns), the
  // quad's 64-float slots from its first warp's prefix fold on, in segment order.
  const int nunit = fold_n * 16;
  for (int idx = threadIdx.x; idx < nunit; idx += blockDim.x) {
    const PendFold& f = pend_info[fold_ref[idx >> 4]];
    const int col = 4 * (idx & 15);
    if (col >= f.cols) continue;  // ragged last quad
    if (!dbg_ok(p.status, f.first >= 0 && f.first + f.nslot <= I)) continue;
    const int nslot = f.nslot;
    const float4* part = reinterpret_cast<const float4*>(p.partials + f.first * 64 + col);
    const uint32_t r0 = residual2<NORM>(p, f.n0 + col), r1 = residual2<NORM>(p, f.n0 + col + 2);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < nslot; s0 += 8) {  // 8 slots in flight, then fold in order
      float4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        v[k] = (s0 + k < nslot) ? __ldcg(part + static_cast<long long>(s0 + k) * 16) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (s0 + k < nslot) {
          if (s0 + k == 0) {
            acc = v[k];
          } else {
            acc.x += v[k].x; acc.y += v[k].y; acc.z += v[k].z; acc.w += v[k].w;
          }
        }
      }
    }
    uint32_t* yo = reinterpret_cast<uint32_t*>(f.y + col);
    yo[0] = emit2<NORM>(acc.x, acc.y, r0);
    yo[1] = emit2<NORM>(acc.z, acc.w, r1);
  }
}

// ----------------------------------------------------------------- prep kernel

// A group of one x row staged in shared memory (272 bytes: the eight lane
// quads of a warp reading eight staged rows land on distinct banks).
constexpr int kStageStride = kGroup * 2 + 16;

// Lane class c of one (group, x row) package row, built by four consecutive
// lanes (lane & ~3 .. + 3, one per class), which agree on the row's scale 2^s
// from the largest magnitude among their 128 values: x' = x 2^s as fp16 pairs
// in operand order go to dst + 80 c (64 bytes), and lane c == 0 writes the
// row's (X_g, f), f = 2^-s, to tail[0..1].  xg: the row's 128 values of
// the group, or nullptr for a zero row (then the row is written as zeros);
// dst == nullptr writes nothing.  Every lane of the warp must call it (it
// shuffles).
// The 16 bf16 pairs of lane class c of one (group, x row), in operand order:
// words 2i, 2i + 1 hold x[16i + 2c], x[16i + 2c + 1] and x[16i + 2c + 8],
// x[16i + 2c + 9].  xg: the row's 128 values of the group, or nullptr for a
// zero row.
template <bool kSharedX = false>
__device__ __forceinline__ void load_row_class(const uint16_t* xg, int c, uint32_t (&w)[16]) {
  if (xg == nullptr) {
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = 0u;
    return;
  }
  // x rows start 4-byte aligned (K even, x 4-byte aligned): one 32-bit load
  // per operand pair; from global memory through L2, since x may be the
  // output of the kernel this one was launched behind
  const uint32_t* xr = reinterpret_cast<const uint32_t*>(xg);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if constexpr (kSharedX) {  // x staged in this CTA's shared memory
      w[2 * i] = xr[8 * i + c];
      w[2 * i + 1] = xr[8 * i + c + 4];
    } else {
      w[2 * i] = __ldcg(xr + 8 * i + c);
      w[2 * i + 1] = __ldcg(xr + 8 * i + c + 4);
    }
  }
}

// Lane class c of one (group, x row) package row from its loaded words, built
// by four consecutive lanes (lane & ~3 .. + 3, one per class), which agree on
// the row's scale 2^s from the largest magnitude among their 128 values:
// x' = x 2^s as fp16 pairs in operand order go to dst + 80 c (64 bytes), and
// lane c == 0 writes the row's (X_g, f), f = 2^-s, to tail[0..1].  dst ==
// nullptr writes nothing.  Every lane of the warp must call it (it shuffles).
__device__ __forceinline__ void finish_row_class(const uint32_t (&w)[16], int c, int lane, uint8_t* dst,
                                                 float* tail) {
  float X = 0.f;       // sum of this lane's 32 values
  uint32_t mag2 = 0u;  // per-half maxima of |x| bits
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    X = (((X + bf16_lo(w[2 * i])) + bf16_hi(w[2 * i])) + bf16_lo(w[2 * i + 1])) + bf16_hi(w[2 * i + 1]);
    mag2 = __vmaxu2(mag2, __vmaxu2(w[2 * i] & 0x7FFF7FFFu, w[2 * i + 1] & 0x7FFF7FFFu));
  }
  uint32_t amax = max(mag2 & 0xFFFFu, mag2 >> 16);  // largest |x| as bf16 magnitude bits
  amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  // biased exponent e of the row's largest |x|: x 2^(141 - e) lies in
  // [2^14, 2^15); the cap keeps 2^s a normal fp32 for zero or tiny rows.
  const int sft = min(141 - static_cast<int>(amax >> 7), 126);
  const float up = __int_as_float((127 + sft) << 23);
  const float f = __int_as_float((127 - sft) << 23);
  if (dst != nullptr) {
    uint32_t h[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 v = fmul2(make_float2(bf16_lo(w[i]), bf16_hi(w[i])), make_float2(up, up));
      asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h[i]) : "f"(v.y), "f"(v.x));  // (hi, lo)
    }
    uint4* o = reinterpret_cast<uint4*>(dst + c * 80);
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
  }
  // group sum of the row: ((X_0 + X_1) + X_2) + X_3 over its four lane classes
  const float X0 = __shfl_sync(0xffffffffu, X, lane & ~3);
  const float X1 = __shfl_sync(0xffffffffu, X, (lane & ~3) + 1);
  const float X2 = __shfl_sync(0xffffffffu, X, (lane & ~3) + 2);
  const float X3 = __shfl_sync(0xffffffffu, X, (lane & ~3) + 3);
  if (c == 0 && dst != nullptr) {
    tail[0] = ((X0 + X1) + X2) + X3;
    tail[1] = f;
  }
}

// load_row_class + finish_row_class (xg == nullptr: a zero row).
__device__ __forceinline__ void build_row_class(const uint16_t* xg, int c, int lane, uint8_t* dst, float* tail) {
  uint32_t w[16];
  load_row_class(xg, c, w);
  finish_row_class(w, c, lane, dst, tail);
}

// The prep kernels run on a 2-D grid, blockIdx.y = matrix, so no CTA
// searches the matrix table (each lookup in the kernel parameters is an L2
// round trip when it misses the constant cache).

// M >= 2: one group per warp; lane (row, c) builds rows `row`
// (and row + 8 for the 16-row package) / lane class c of the group's
// activation package (rows >= M are zeros).
template <int MODE, int MAXMAT>
__global__ void __launch_bounds__(256) prep_kernel(const __grid_constant__ StreamParams<MAXMAT> p) {
  // Launched early behind the previous kernel of the stream (programmatic
  // dependent launch): the next kernel may launch at once, but nothing here
  // is touched before the previous one has finished -- it may still read the
  // workspace, or write this call's x.
  grid_dependents_launch();
  grid_dependency_wait();
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *p.status = 0u;
  constexpr int kRows = Pkg<MODE>::kRows;
  const MatParams& m = mat(p, blockIdx.y);
  // M >= 2 takes no tickets.  For the per-quad reduce their array holds each
  // quad's matrix instead (a load from it replaces a search of the matrix
  // table); for the per-warp reduce the streaming warps' split-quad records
  // are cleared, over the whole grid.
  if constexpr (MAXMAT > 1) {
    if (p.per_warp_reduce) {
      const int nthr = gridDim.x * gridDim.y * blockDim.x;
      for (int i = (blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x; i < p.W; i += nthr)
        p.recs[i] = 0ull;
    } else {
      const int nq = div_up(m.N, kQuadTiles * kTileN);
      for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nq; i += gridDim.x * blockDim.x)
        p.tickets[m.quad_begin + i] = blockIdx.y;
    }
  }
  const int G = m.K / kGroup;
  const int lane = threadIdx.x & 31;
  const int row = lane >> 2, c = lane & 3;
  const int nwarp = blockDim.x >> 5;
  // A warp's group: its M rows of x are staged in shared memory with 16-byte
  // loads (rows kStageStride bytes apart: the eight lane quads then read
  // eight rows on distinct banks), then built from there -- the same words
  // as reading them from global memory one by one, in a quarter of the load
  // instructions (layer step M = 8 42.6 -> 41.8 us, M = 16 68.9 -> 67.6 us).
  // x only 4-byte aligned is read directly.
  __shared__ __align__(16) uint8_t xs[8][kRows][kStageStride];
  const bool staged = (reinterpret_cast<uintptr_t>(m.x) & 15u) == 0;
  const int wp = threadIdx.x >> 5;
  for (int g = nwarp * blockIdx.x + wp; g < G; g += nwarp * gridDim.x) {
    uint8_t* out = m.xpkg + static_cast<long long>(g) * Pkg<MODE>::kBytes;
    float* tail = reinterpret_cast<float*>(out + kRows * Pkg<MODE>::kRowBytes);
    if (staged) {
      for (int j = lane; j < p.M * 16; j += 32) {
        const int rr = j >> 4, part = j & 15;
        const uint4 v = __ldcg(reinterpret_cast<const uint4*>(m.x + static_cast<long long>(rr) * m.K + kGroup * g) + part);
        *reinterpret_cast<uint4*>(&xs[wp][rr][part * 16]) = v;
      }
      __syncwarp();
#pragma unroll
      for (int row8 = 0; row8 < kRows; row8 += 8) {
        const int rw = row8 + row;
        uint32_t w[16];
        load_row_class<true>(rw < p.M ? reinterpret_cast<const uint16_t*>(&xs[wp][rw][0]) : nullptr, c, w);
        finish_row_class(w, c, lane, out + rw * Pkg<MODE>::kRowBytes, tail + 2 * rw);
      }
      __syncwarp();  // the rows are read before the next group's overwrite them
    } else {
#pragma unroll
      for (int row8 = 0; row8 < kRows; row8 += 8) {
        const int rw = row8 + row;
        build_row_class(rw < p.M ? m.x + static_cast<long long>(rw) * m.K + kGroup * g : nullptr, c, lane,
                        out + rw * Pkg<MODE>::kRowBytes, tail + 2 * rw);
      }
    }
  }
}

// M = 1: the one-row package needs four lanes, so a warp
// builds eight groups at once, lane (j, c) class c of group 8 k + j of its
// share.  One-warp CTAs with few registers fit on an SM beside a streaming
// CTA: the next call's prep is resident before the previous call has ended,
// and never holds an SM the streaming kernel needs.  Also clears the
// split-quad tickets and the status word.
template <int MODE, int MAXMAT>
__global__ void __launch_bounds__(32) prep1_kernel(const __grid_constant__ StreamParams<MAXMAT> p) {
  grid_dependents_launch();
  grid_dependency_wait();  // as in prep_kernel
  const int lane = threadIdx.x;
  const MatParams& m = mat(p, blockIdx.y);
  const int G = m.K / kGroup;
  // this matrix's split-quad tickets
  const int nq = div_up(m.N, kQuadTiles * kTileN);
  for (int i = blockIdx.x * 32 + lane; i < nq; i += gridDim.x * 32) p.tickets[m.quad_begin + i] = 0u;
  if (blockIdx.x == 0 && blockIdx.y == 0 && lane == 0) *p.status = 0u;
  const int j = lane >> 2, c = lane & 3;
  for (int base = 8 * blockIdx.x; base < G; base += 8 * gridDim.x) {  // warp-uniform trip count
    const int g = base + j;
    const bool in = g < G;
    uint8_t* out = in ? m.xpkg + static_cast<long long>(g) * Pkg<MODE>::kBytes : nullptr;
    build_row_class(in ? m.x + kGroup * g : nullptr, c, lane, out, reinterpret_cast<float*>(out + Pkg<MODE>::kRowBytes));
  }
}

// ----------------------------------------------------------------- M = 1 with CTA-local packages

// A call at M = 1 whose CTAs' working sets fit in shared memory runs without
// the prep kernel ("local" calls):
//  * each CTA stages, after its dependency wait, the groups of x its warps
//    need (16-byte cp.async copies by every thread, at a 272-byte stride per
//    group so that the lanes reading them hit distinct banks) and builds
//    those groups' activation packages in its own shared memory, with exactly
//    the prep kernel's arithmetic (load_row_class, finish_row_class), so
//    every bit matches; the staging sits at the far end of the package area
//    and is converted in place, pass by pass;
//  * the ring slots carry weights only, and every slot is filled before the
//    dependency wait;
//  * a split quad whose segments all lie in this CTA's item range is folded
//    from shared-memory partial slots at the CTA's end; a quad that begins in
//    this CTA and continues in the next gets this CTA's left fold of its
//    segments stored as one global slot; the segments of a quad that began in
//    an earlier CTA go to global slots one by one; fold1_kernel, launched
//    behind the streaming kernel, folds those boundary quads once every CTA
//    has finished (one bulk copy pulls each quad's slots).  The fold order is
//    the left fold over segments either way.
// This removes a dependent kernel (prep -> stream) from every call.  Calls
// whose CTAs would need more shared memory than is free (e.g. the whole
// decode step of hundreds of matrices) or whose x is not 16-byte aligned take
// the prep-kernel path.  (Folding the boundary quads inside the streaming
// kernel instead, through tickets, was measured slower: the fence and the
// atomic round trips behind every CTA's stream cost more than the fold
// kernel's launch.)

constexpr int kLocalMaxEntries = 8;                       // matrices one CTA's range may touch
constexpr int kLocalSlot = kQuadTiles * kBlockBytes;      // ring slot: weights only (4352 bytes)
constexpr int kLocalSlots = 2 * kNW;                      // ring slots per CTA: 2 per warp at 16 warps
constexpr int kLocalBarBytes = 512;                       // ring mbarriers (32 x 8)
constexpr int kLocalRing = kLocalSlots * kLocalSlot;      // slot d of warp w at (d * warps + w)
constexpr int kLocalDyn = 232448 - 4096;                  // dynamic shared memory (static use stays below 4 KB)
constexpr int kLocalSpace = kLocalDyn - kLocalBarBytes - kLocalRing;  // packages + partial slots
constexpr int kPkg1 = Pkg<kMMA1>::kBytes;                 // one M = 1 package (336 bytes)
constexpr int kMaxFoldSlots = 65536 / (kGroup * kSegGroups) + 1;  // slots of one boundary fold, at most
constexpr int kFoldSmem = kMaxFoldSlots * 64 * 4 + 16;    // fold1_kernel: the slots and an mbarrier
static_assert(kLocalSpace > 0 && kLocalRing % 128 == 0, "local layout");

// The groups of matrix mi that a CTA's items touch, and where their packages
// sit in the CTA's package area.
struct LocalEntry {
  int mi, g_lo, g_hi, pkg;
};

// Groups [g_lo, g_hi) needed by local items [lo, hi) of one matrix (S
// segments per quad, G groups): the items' segments when they stay within
// one quad, every group when they cross a quad boundary.
__host__ __device__ inline void local_groups(long long lo, long long hi, int S, int G, int& g_lo, int& g_hi) {
  const long long qa = lo / S, qb = (hi - 1) / S;
  if (qa == qb) {
    g_lo = static_cast<int>(lo - qa * S) * kSegGroups;
    const int e = static_cast<int>(hi - 1 - qb * S) * kSegGroups + kSegGroups;
    g_hi = e < G ? e : G;
  } else {
    g_lo = 0;
    g_hi = G;
  }
}

// The table of a CTA whose items are [A, B) (A < B): returns the number of
// entries (-1 if more than kLocalMaxEntries) and the total package count.
// `at` gives item_begin(i), K(i), N(i) of matrix i; the host and the device
// build the same table from it.
#pragma nv_exec_check_disable
template <class MatAt>
__host__ __device__ inline int local_table(long long A, long long B, int count, const MatAt& at, LocalEntry* t,
                                           int& npkg) {
  int lo = 0, hi = count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (at.begin(mid) <= A) lo = mid; else hi = mid - 1;
  }
  int n = 0;
  npkg = 0;
  for (int mi = lo; mi < count && at.begin(mi) < B; ++mi) {
    if (n == kLocalMaxEntries) return -1;
    const int G = at.K(mi) / kGroup, S = div_up(G, kSegGroups), NQ = div_up(at.N(mi), kQuadTiles * kTileN);
    const long long b0 = at.begin(mi), b1 = b0 + static_cast<long long>(NQ) * S;
    const long long lo_it = (A > b0 ? A : b0) - b0, hi_it = (B < b1 ? B : b1) - b0;
    LocalEntry& e = t[n++];
    e.mi = mi;
    local_groups(lo_it, hi_it, S, G, e.g_lo, e.g_hi);
    e.pkg = npkg;
    npkg += e.g_hi - e.g_lo;
  }
  return n;
}

template <int MAXMAT>
struct DevMats {
  const StreamParams<MAXMAT>& p;
  __device__ long long begin(int i) const { return mat(p, i).item_begin; }
  __device__ int K(int i) const { return mat(p, i).K; }
  __device__ int N(int i) const { return mat(p, i).N; }
};

// The status word of a local call is 64 bits: the code in bits 0..7 (what
// w4g128_workspace_status reports) and, above it, a tag of the streaming
// grid that wrote it.  A call clears the word when it starts (CTA 0, after
// its dependency wait) and records a failure at any time; both are
// compare-and-swap loops on the tag, so a failure recorded by another CTA of
// the same grid before the clear survives it, and a stale or uninitialised
// word is replaced.  (Replays of one CUDA graph node share their %gridid and
// so their tag: a failure of one replay stays reported by the next.)
__device__ __forceinline__ unsigned long long grid_tag() {
  unsigned long long g;
  asm volatile("mov.u64 %0, %%gridid;" : "=l"(g));
  // a multiplicative hash (odd constant: a bijection), so that small launch
  // numbers do not look like words with zero upper bytes
  return ((g + 1ull) * 0x9E3779B97F4A7C15ull) >> 8;
}

__device__ __forceinline__ void status_begin(unsigned* status) {
  auto* st = reinterpret_cast<unsigned long long*>(status);
  const unsigned long long tag = grid_tag();
  unsigned long long cur = ld_relaxed_u64(st);
  while ((cur >> 8) != tag) {
    const unsigned long long prev = atomicCAS(st, cur, tag << 8);
    if (prev == cur) return;
    cur = prev;
  }
}

__device__ __forceinline__ void status_fail(unsigned* status, unsigned code) {
  auto* st = reinterpret_cast<unsigned long long*>(status);
  const unsigned long long tag = grid_tag();
  unsigned long long cur = ld_relaxed_u64(st);
  while (!((cur >> 8) == tag && (cur & 0xFFull) != 0ull)) {
    const unsigned long long prev = atomicCAS(st, cur, (tag << 8) | code);
    if (prev == cur) return;
    cur = prev;
  }
}

// cond, or (debug builds) false after recording the failure in a local
// call's tagged status word.
__device__ __forceinline__ bool dbg_ok_local(unsigned* status, bool cond) {
  if constexpr (kDebug) {
    if (!cond) status_fail(status, W4G128_ERR_INTERNAL);
    return cond;
  } else {
    return true;
  }
}

// Debug builds: a chunk's weight blocks lie inside their matrix's packed bytes.
template <int MAXMAT>
__device__ __forceinline__ bool weights_in_range(const StreamParams<MAXMAT>& p, const Cursor& c) {
  if constexpr (!kDebug) {
    return true;
  } else {
    const MatParams& m = mat(p, c.mi);
    return dbg_ok_local(p.status, c.src >= m.packed &&
                                      c.src + c.ntiles * kBlockBytes <= m.packed + packed_bytes_of(m.K, m.N));
  }
}

// A fold the CTA does at its end: slots [first, first + nslot) of its
// shared-memory partial area (indices relative to its first item), written
// to y (a quad inside the CTA's range) or, for the quad that continues into
// the next CTA, stored as one global partial slot.
struct LocalFold {
  long long first;  // first slot (CTA item index)
  uint16_t* y;      // the quad's first output column (internal), or nullptr
  float* gslot;     // the global slot for the CTA's prefix fold (boundary), or nullptr
  int nslot;
  int cols;
  int n0;
  int pad;
};

// CTAs of 13-16 warps: the several-matrix forms (a decoder layer's step)
// take 128 registers, a 16-warp CTA then holding the SM's whole register
// file, and interleave a quad's tiles in pairs (spilling a few words); the
// one-matrix form keeps 120 registers and goes tile by tile, which leaves
// room for fold1_kernel's small CTAs beside the stream.  Measured on one
// GPU: the layer step 36.70 -> 36.40 us with the pairs, the 5120x248320
// lm_head 101.9 -> 103.7 us.  The WIDE form (CTAs of at most kWideWarps
// warps: calls too small to give every SM 16 warps) takes 168 registers and
// interleaves all four tiles, since there a warp is often alone on its
// scheduler.
template <int MAXMAT, bool NORM, bool WIDE>
__global__ void __maxnreg__(WIDE ? 168 : (MAXMAT == 1 ? 120 : 128))
    stream1_local_kernel(const __grid_constant__ StreamParams<MAXMAT> p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int NA = Acc<kMMA1>::kN;
  __shared__ LocalEntry tbl[kLocalMaxEntries];
  __shared__ int tbl_n, tbl_npkg;
  __shared__ int fold_n;
  __shared__ LocalFold folds[2 * kNW];
  __shared__ int fold_fail;

  // Paired quads (one matrix): CTA 2q (the leader, cluster rank 0) streams
  // the first half of quad q's segments and CTA 2q + 1 the rest; at the end
  // the partner stores its segment sums into the leader's partial slots and
  // the leader folds all of them in segment order.  Every thread of both CTAs
  // arrives here and passes the two cluster barrier phases below on every path.
  const bool pair = MAXMAT == 1 && p.pair != 0;
  if (pair) cluster_arrive_relaxed();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, c = lane & 3;
  const int cw = blockDim.x >> 5;
  // a CTA's 32 ring slots are shared out among its warps: 2 each at 16 warps,
  // up to 8 each in smaller CTAs, whose warps then keep more bytes in flight
  const int D = p.depth;
  const int wg = blockIdx.x * cw + warp;
  const long long I = p.total_items;
  // The CTA's items [A, B): from the host's table (calls of up to
  // kFewMatrices matrices), else the balanced split.
  long long A, B;
  if constexpr (MAXMAT <= kFewMatrices) {
    A = p.cta_begin[blockIdx.x];
    B = p.cta_begin[blockIdx.x + 1];
  } else {
    A = split_at(I, static_cast<long long>(blockIdx.x) * cw, p.W);
    B = split_at(I, min((static_cast<int>(blockIdx.x) + 1) * cw, p.W), p.W);
  }
  // With the table, warp w of the CTA streams [A + n w / cw, A + n (w + 1) / cw),
  // n = B - A; the last item of the warp that holds item i of [A, B):
  const unsigned n_cta = static_cast<unsigned>(B - A);
  auto warp_first = [&](int w) -> long long {
    if constexpr (MAXMAT <= kFewMatrices) return A + static_cast<long long>(n_cta * static_cast<unsigned>(w) / cw);
    else return split_at(I, static_cast<long long>(blockIdx.x) * cw + w, p.W);
  };
  auto owner_last = [&](long long i) -> long long {
    if constexpr (MAXMAT <= kFewMatrices) {
      const int wo = static_cast<int>((static_cast<unsigned>(i - A + 1) * cw - 1u) / n_cta);
      return warp_first(wo + 1) - 1;
    } else {
      return split_at(I, owner_of(i, I, p.W) + 1, p.W) - 1;
    }
  };
  const uint32_t bars = smem_addr(smem);
  const uint32_t ring0 = bars + kLocalBarBytes;
  uint8_t* const pkg_area = smem + p.local_pkg_off;
  float* const part_area = reinterpret_cast<float*>(smem + p.local_part_off);
  // the pair's items [Aq, Bq): one quad, whose slots all sit in the leader
  long long Aq = A, Bq = B;
  if constexpr (MAXMAT <= kFewMatrices) {
    if (pair && (gridDim.x & 1u) == 0u && gridDim.x <= static_cast<unsigned>(kMaxLocalCtas)) {
      Aq = p.cta_begin[blockIdx.x & ~1u];
      Bq = p.cta_begin[(blockIdx.x | 1u) + 1u];
    }
  }
  // the slots this CTA's folds may read
  const long long slot_cap = pair ? Bq - Aq : B - A;

  if (threadIdx.x == 0) {
    fold_n = 0;
    fold_fail = 0;
    int np = 0;
    tbl_n = local_table(A, B, p.count, DevMats<MAXMAT>{p}, tbl, np);
    tbl_npkg = np;
  }
  if (lane == 0) {
    for (int d = 0; d < D; ++d) mbar_init(bars + 8 * (warp * D + d), 1);
    fence_mbar_init();
  }
  __syncthreads();
  // The host launches this kernel only for M = 1 calls whose every CTA fits
  // (the same table function); a CTA that does not fit records the error and
  // touches nothing.
  // A pair must be CTAs 2q, 2q + 1 of a two-CTA cluster holding exactly the
  // segments of one quad, in that order, with room for all of them in the
  // leader (both CTAs take the same decision from the same words).
  const bool pair_bad =
      pair && ((gridDim.x & 1u) != 0u || cluster_nctarank() != 2u || cluster_ctarank() != (blockIdx.x & 1u) ||
               Aq < 0 || Bq > I || Bq - Aq != div_up(mat(p, 0).K / kGroup, kSegGroups) ||
               (Aq - mat(p, 0).item_begin) % (Bq - Aq) != 0 || A < Aq || B > Bq ||
               p.local_part_off + (Bq - Aq) * 64 * 4 > kLocalDyn);
  if (pair_bad || tbl_n <= 0 || p.M != 1 || p.local_pkg_off != kLocalBarBytes + kLocalRing || D < 2 ||
      D * cw > kLocalSlots || A < 0 || B < A || B > I || (B - A) * cw >= (1ll << 31) ||
      p.local_pkg_off + static_cast<long long>(tbl_npkg) * kPkg1 > p.local_part_off ||
      p.local_part_off + (B - A) * 64 * 4 > kLocalDyn) {
    if (threadIdx.x == 0) status_fail(p.status, W4G128_ERR_INTERNAL);
    if (pair) {  // the partner CTA still passes both phases
      cluster_wait_acquire();
      cluster_arrive_release();
      cluster_wait_acquire();
    }
    return;
  }
  const int mi_a = tbl[0].mi;
  const int npkg = tbl_npkg;
  // x of the CTA's package t is staged at stage + t * kStageStride, at the far
  // end of the package area (package t is built at pkg_area + t * kPkg1)
  uint8_t* const stage = pkg_area + static_cast<long long>(npkg) * (kPkg1 - kStageStride);
  // package of (matrix mi, group g) in the CTA's package area
  auto local_pkg = [&](int mi, int g) -> const uint8_t* {
    const LocalEntry& e = tbl[mi - mi_a];
    return pkg_area + static_cast<long long>(e.pkg + g - e.g_lo) * kPkg1;
  };

  const long long it_a = warp_first(warp), it_b = warp_first(warp + 1);
  const bool streams = (MAXMAT <= kFewMatrices) ? it_a < it_b : wg < p.W;
  uint64_t pol_w = 0;
  Cursor cc, ic;
  unsigned issued = 0u;
  // the weights of chunk ic into this warp's ring slot d (lane 0 issues)
  auto issue_into = [&](int d) {
    if (lane == 0) {
      const uint32_t sa = ring0 + (d * cw + warp) * kLocalSlot, ba = bars + 8 * (warp * D + d);
      if (weights_in_range(p, ic)) {
        mbar_arrive_expect_tx(ba, ic.ntiles * kBlockBytes);
        bulk_g2s(sa, ic.src, ic.ntiles * kBlockBytes, ba, pol_w);
      } else {
        mbar_arrive_plain(ba);
      }
    }
    cursor_next<kMMA1>(ic, p);
    ++issued;
  };
  if (streams) {
    if (lane == 0) pol_w = l2_policy_evict_first();
    cursor_seek<kMMA1>(cc, p, it_a);
    ic = cc;
    // The weights do not depend on earlier work: start them now.  A small
    // CTA (WIDE) fills its whole ring; a 16-warp CTA issues one chunk per
    // warp and the rest after the wait: a deeper start competes with the
    // previous call's last CTAs for HBM (measured on back-to-back layer
    // steps: 38.5 us with the ring filled early, 37.8 with one chunk).
    const unsigned early = WIDE ? static_cast<unsigned>(D) : 1u;
    while (issued < early && ic.item < it_b) issue_into(static_cast<int>(issued));
  }
  grid_dependency_wait();  // the previous kernel has finished: x is final, the workspace free
  grid_dependents_launch();  // the boundary fold may launch; it waits for this grid
  if (streams) {  // the rest of the ring
    while (issued < static_cast<unsigned>(D) && ic.item < it_b) issue_into(static_cast<int>(issued));
  }

  // ---- stage x (16-byte cp.async copies by every thread), then build the packages
  for (int idx = threadIdx.x; idx < npkg * 16; idx += blockDim.x) {
    const int t = idx >> 4, part = idx & 15;
    int e = 0;
    while (e + 1 < tbl_n && tbl[e + 1].pkg <= t) ++e;
    const int g = tbl[e].g_lo + (t - tbl[e].pkg);
    if (dbg_ok_local(p.status, g >= 0 && g < mat(p, tbl[e].mi).K / kGroup))
      cp_async16(smem_addr(stage + t * kStageStride + part * 16),
                 mat(p, tbl[e].mi).x + static_cast<long long>(g) * kGroup + part * 8);
  }
  cp_async_wait_all();
  // the status word is cleared by a thread of the second warp (thread 0 of a
  // one-warp CTA)
  if (blockIdx.x == 0 && threadIdx.x == (blockDim.x > 32 ? 32u : 0u)) status_begin(p.status);
  __syncthreads();  // x staged
  {
    // lanes (j, c): lane class c of package base + j, eight packages per warp
    // per pass; each pass reads its staged groups into registers, then (after
    // a barrier) overwrites the bytes below the next pass's staging
    const int npass = div_up(npkg, 8 * cw);
    for (int ps = 0; ps < npass; ++ps) {
      const int t = ps * 8 * cw + 8 * warp + (lane >> 2);
      const bool in = t < npkg;
      uint32_t wx[16];
      load_row_class<true>(in ? reinterpret_cast<const uint16_t*>(stage + t * kStageStride) : nullptr, c, wx);
      __syncthreads();
      uint8_t* out = in ? pkg_area + static_cast<long long>(t) * kPkg1 : nullptr;
      finish_row_class(wx, c, lane, out, reinterpret_cast<float*>(out + Pkg<kMMA1>::kRowBytes));
    }
  }
  __syncthreads();  // packages written

  bool failed = false;
  float seg[kQuadTiles][NA], tot[kQuadTiles][NA];
  int n_pend = 0;
  if (streams) {
    cc.xsrc = local_pkg(cc.mi, cc.g);
#pragma unroll
    for (int t = 0; t < kQuadTiles; ++t)
#pragma unroll
      for (int e = 0; e < NA; ++e) seg[t][e] = tot[t][e] = 0.f;

    unsigned done = 0;
    int slot = 0;
    uint32_t parity = 0u;
    while (cc.item < it_b) {
      if (!mbar_wait_bounded(bars + 8 * (warp * D + slot), parity, p.wait_ns)) {
        if (lane == 0) {
          status_fail(p.status, W4G128_ERR_TIMEOUT);
          for (unsigned k = done + 1; k < issued; ++k)
            (void)mbar_wait_bounded(bars + 8 * (warp * D + static_cast<int>(k % D)), (k / D) & 1u, p.wait_ns);
        }
        __syncwarp();
        failed = true;
        break;
      }
      const int ntiles = cc.ntiles;
      const uint8_t* sl = smem + kLocalBarBytes + (slot * cw + warp) * kLocalSlot;
      compute_chunk<kMMA1, WIDE ? 2 : (MAXMAT == 1 ? 0 : 1)>(sl, cc.xsrc, ntiles, lane, seg);
      __syncwarp();
      if (ic.item < it_b) {
        if (lane == 0) fence_proxy_async_smem();  // the slot's reads are done before the copy rewrites it
        issue_into(slot);
      }
      ++done;
      if (++slot == D) {
        slot = 0;
        parity ^= 1u;
      }

      if (cc.g + 1 == cc.g_end) {
        // ---- end of a segment
        const MatParams& m = mat(p, cc.mi);
        const int S = cc.S;
        const long long q_first = m.item_begin + static_cast<long long>(cc.q) * S;
        const long long q_last = q_first + S - 1;
        const bool owned = (q_first >= it_a) && (q_last < it_b);
        const bool prefix = (q_first >= it_a) && !owned;
        if (owned || prefix) {
#pragma unroll
          for (int t = 0; t < kQuadTiles; ++t)
#pragma unroll
            for (int e = 0; e < NA; ++e) tot[t][e] = (cc.s == 0) ? seg[t][e] : tot[t][e] + seg[t][e];
        }
        if (!owned && (!prefix || cc.item + 1 == it_b) && dbg_ok_local(p.status, cc.item >= A && cc.item < B)) {
          // a quad that began before this CTA: the segment sum goes to its
          // global slot for the boundary fold; otherwise to this CTA's slot
          // (a pair's partner keeps its slots in shared memory for the leader)
          float* part = (q_first < A && !pair) ? p.partials + cc.item * 64 : part_area + (cc.item - A) * 64;
          if (c == 0) {
#pragma unroll
            for (int t = 0; t < kQuadTiles; ++t) {
              if (t < ntiles) {
                part[16 * t + r] = prefix ? tot[t][0] : seg[t][0];
                part[16 * t + r + 8] = prefix ? tot[t][1] : seg[t][1];
              }
            }
          }
        }
#pragma unroll
        for (int t = 0; t < kQuadTiles; ++t)
#pragma unroll
          for (int e = 0; e < NA; ++e) seg[t][e] = 0.f;

        const bool quad_end = (cc.s == S - 1) || (cc.item + 1 == it_b);
        if (quad_end) {
          const int n0 = kQuadTiles * kTileN * cc.q;
          if (owned && dbg_ok_local(p.status, n0 + kTileN * ntiles <= m.N)) {
            if (c == 0) {
#pragma unroll
              for (int t = 0; t < kQuadTiles; ++t) {
                if (t < ntiles) {
                  const int n = n0 + 16 * t + r;
                  m.y[n] = emit<NORM>(p, n, tot[t][0]);
                  m.y[n + 8] = emit<NORM>(p, n + 8, tot[t][1]);
                }
              }
            }
          } else if (q_first >= A && n_pend < 2 && (cc.s == S - 1 || (q_last >= B && cc.item + 1 == B))) {
            // this warp holds the last segment of a quad inside the CTA's
            // range (fold it to y), or the CTA's last item inside a quad that
            // continues in the next CTA (fold the CTA's share to one global slot)
            if (lane == 0) {
              const long long first = owner_last(q_first);
              LocalFold& f = folds[atomicAdd(&fold_n, 1)];
              const bool inner = cc.s == S - 1 || pair;  // a pair's leader folds the whole quad
              f.first = first - A;
              f.nslot = static_cast<int>((inner ? q_last : B - 1) + 1 - first);
              f.y = inner ? m.y + n0 : nullptr;
              f.gslot = inner ? nullptr : p.partials + (B - 1) * 64;
              f.cols = kTileN * ntiles;
              f.n0 = n0;
            }
            ++n_pend;
          }
        }
      }
      cursor_next<kMMA1>(cc, p);
      if (cc.g == 0 && cc.item < it_b) cc.xsrc = local_pkg(cc.mi, 0);
    }
    if (failed && lane == 0) atomicOr(&fold_fail, 1);
  }
  __syncthreads();  // every warp's slots are written
  if (pair) {
    cluster_wait_acquire();  // both CTAs of the pair have started: the leader's shared memory is there
    if (blockIdx.x & 1u) {   // the partner: its slots to the leader's, after the leader's own
      const uint32_t dst = cluster_map(smem_addr(part_area), 0u) + static_cast<uint32_t>(A - Aq) * 256u;
      const float4* src = reinterpret_cast<const float4*>(part_area);
      const int n16 = static_cast<int>(B - A) * 16;
      for (int i = threadIdx.x; i < n16; i += blockDim.x) st_cluster_v4(dst + 16u * i, src[i]);
    }
    cluster_arrive_release();
    cluster_wait_acquire();  // the partner's slots are in the leader's shared memory
  }
  if (fold_fail) return;  // a timed-out warp left its quads unreduced (the status word says so)

  // ---- the CTA's folds: one thread per (fold, 4 columns), slots in order
  const int nunit = fold_n * 16;
  for (int idx = threadIdx.x; idx < nunit; idx += blockDim.x) {
    const LocalFold& f = folds[idx >> 4];
    const int col = 4 * (idx & 15);
    if (col >= f.cols) continue;
    if (!dbg_ok_local(p.status, f.first >= 0 && f.first + f.nslot <= slot_cap)) continue;
    const float4* part = reinterpret_cast<const float4*>(part_area + f.first * 64 + col);
    uint32_t r0 = 0u, r1 = 0u;
    if (f.y != nullptr) {
      r0 = residual2<NORM>(p, f.n0 + col);
      r1 = residual2<NORM>(p, f.n0 + col + 2);
    }
    float4 acc = part[0];
    for (int k = 1; k < f.nslot; ++k) {
      const float4 v = part[static_cast<long long>(k) * 16];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    if (f.y != nullptr) {
      uint32_t* yo = reinterpret_cast<uint32_t*>(f.y + col);
      yo[0] = emit2<NORM>(acc.x, acc.y, r0);
      yo[1] = emit2<NORM>(acc.z, acc.w, r1);
    } else {
      *reinterpret_cast<float4*>(f.gslot + col) = acc;
    }
  }
}

// The boundary quads of a local call: for each boundary cb between streaming
// CTAs cb - 1 and cb whose first item lies inside a quad that began in CTA
// cb - 1, fold that quad's slots -- CTA cb - 1's fold of its share, then the
// later segments one by one, a contiguous run -- once the streaming grid has
// finished.  A quad spanning more CTAs is folded at its first boundary only.
// One 32-thread CTA per boundary: lane 0 pulls the run into shared memory
// with one bulk copy, lanes 0..15 fold one 4-column unit each.
template <int MAXMAT, bool NORM>
__global__ void __launch_bounds__(32) fold1_kernel(const __grid_constant__ StreamParams<MAXMAT> p) {
  extern __shared__ __align__(128) uint8_t fsm[];
  // the next kernel may launch now; it waits for this grid, which does not
  // finish before the streaming grid (the last CTA always waits for it)
  grid_dependents_launch();
  const int cb = blockIdx.x + 1;
  const long long I = p.total_items;
  long long Ac, Ap;
  if constexpr (MAXMAT <= kFewMatrices) {
    Ac = p.cta_begin[cb];
    Ap = p.cta_begin[cb - 1];
  } else {
    Ac = split_at(I, min(static_cast<long long>(cb) * p.cta_warps, static_cast<long long>(p.W)), p.W);
    Ap = split_at(I, static_cast<long long>(cb - 1) * p.cta_warps, p.W);
  }
  int lo = 0;
  if constexpr (MAXMAT > 1) {
    int hi = p.count - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.mats[mid].item_begin <= Ac) lo = mid; else hi = mid - 1;
    }
  }
  const MatParams& m = mat(p, lo);
  const int S = div_up(m.K / kGroup, kSegGroups);
  const long long local = Ac - m.item_begin;
  const int q = static_cast<int>(local / S);
  const int s = static_cast<int>(local - static_cast<long long>(q) * S);
  if (Ac >= I || s == 0 || Ac - s < Ap) {  // no quad begins in CTA cb - 1 and continues here
    if (blockIdx.x + 1 == gridDim.x) grid_dependency_wait();
    return;
  }
  const int nslot = S - s + 1;  // CTA cb - 1's slot (item Ac - 1), then segments s .. S - 1
  if (!dbg_ok_local(p.status, Ac - 1 + nslot <= I && nslot <= kMaxFoldSlots)) {
    if (blockIdx.x + 1 == gridDim.x) grid_dependency_wait();
    return;
  }
  const int cols = kTileN * min(kQuadTiles, m.N / kTileN - kQuadTiles * q);
  const int col = 4 * threadIdx.x;
  const bool active = col < cols && threadIdx.x < 16;
  const int n = kQuadTiles * kTileN * q + col;
  uint32_t r0 = 0u, r1 = 0u;
  if (active) {
    r0 = residual2<NORM>(p, n);
    r1 = residual2<NORM>(p, n + 2);
  }
  uint16_t* y = m.y;
  const uint32_t bar = smem_addr(fsm + kMaxFoldSlots * 64 * 4);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  grid_dependency_wait();  // every slot of the streaming grid is written and visible
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nslot) * 256u);
    bulk_g2s(smem_addr(fsm), p.partials + (Ac - 1) * 64, static_cast<uint32_t>(nslot) * 256u, bar,
             l2_policy_evict_first());
  }
  if (!mbar_wait_bounded(bar, 0u, p.wait_ns)) {
    if (threadIdx.x == 0) status_fail(p.status, W4G128_ERR_TIMEOUT);
    return;
  }
  if (!active) return;
  const float4* part = reinterpret_cast<const float4*>(fsm) + threadIdx.x;
  float4 acc = part[0];
  for (int k = 1; k < nslot; ++k) {
    const float4 v = part[k * 16];
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
  }
  uint32_t* yo = reinterpret_cast<uint32_t*>(y + n);
  yo[0] = emit2<NORM>(acc.x, acc.y, r0);
  yo[1] = emit2<NORM>(acc.z, acc.w, r1);
}

// ----------------------------------------------------------------- reduce kernel

// M >= 2: folds the segment partials of every quad the schedule split between
// warps.  Two forms; a call takes the one with the smaller grid.
//
// Per quad (calls with no more quads than streaming warps): one CTA per
// quad.  The quad's partial slots -- the fold of the segments its first warp
// held, then one slot per later segment -- are one contiguous run of M x 64
// fp32 slots, pulled into shared memory by 1-D bulk copies of up to
// kRedChunk slots (kRedChunkDeep for calls with deep quads whose fold CTAs
// fit one wave at that size; two stages), and each thread folds one (row, 4
// adjacent columns) unit over them in order -- the left fold a single warp
// would have made.  CTAs take quads from the last back when the call's last
// matrix is its deepest.  Quads owned by one warp were written by the
// streaming kernel; their CTAs exit before waiting for it.
constexpr int kMaxRows = W4G128_MAX_M;
constexpr int kRedChunk = 8;                               // segments per bulk copy
constexpr int kRedThreads = kMaxRows * 16;                 // one per (row, 4 columns)
constexpr int kRedStageBytes = kRedChunk * kMaxRows * 64 * 4;  // the largest stage (M = 16)
constexpr int kRedSmem = 2 * kRedStageBytes + 16;          // two stages + two mbarriers, at most
// a call's reduce CTAs: 16 M threads (one per row and 4 columns), two stages of M rows
__host__ __device__ constexpr int red_threads(int M) { return ((16 * M + 31) / 32) * 32; }
__host__ __device__ constexpr int red_smem(int M, int chunk = kRedChunk) { return 2 * chunk * M * 64 * 4 + 16; }
// Calls whose quads are deeper than kRedChunk segments and whose fold CTAs
// all fit one wave at the larger stage copy kRedChunkDeep slots at a time
// (M <= 8; the same shared memory as M = 16 at kRedChunk).
constexpr int kRedChunkDeep = 16;
static_assert(red_smem(8, kRedChunkDeep) <= kRedSmem, "deep stages fit the reduce kernel's shared memory");

template <int MAXMAT, bool NORM>
__global__ void __launch_bounds__(kRedThreads) reduce_quads_kernel(const __grid_constant__ StreamParams<MAXMAT> p) {
  extern __shared__ __align__(128) uint8_t rsm[];
  __shared__ int ok;
  // deepest quads first when the host says they come last (a layer's down
  // projection): their folds take the most copy rounds
  const int gq = p.red_reverse ? p.total_quads - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x);
  int lo = 0;
  if constexpr (MAXMAT > 1) lo = static_cast<int>(__ldcg(p.tickets + gq));  // written by the prep kernel
  const MatParams& m = mat(p, lo);
  const int q = gq - m.quad_begin;
  const int G = m.K / kGroup, S = div_up(G, kSegGroups), T = m.N / kTileN;  // the MMA modes' segments
  const long long I = p.total_items;
  const long long q_first = m.item_begin + static_cast<long long>(q) * S;
  const int wf = owner_of(q_first, I, p.W);
  // The next call's prep kernel may launch now; it waits for this grid to
  // finish, and this grid does not finish before the streaming kernel: every
  // CTA waits for it (below, or here for owned quads).
  grid_dependents_launch();
  if (wf == owner_of(q_first + S - 1, I, p.W)) {  // owned: y is written
    grid_dependency_wait();
    return;
  }
  // Slots from the prefix run's last segment (which holds the fold of the
  // segments before it) to the quad's last segment.
  const long long first = I * (wf + 1) / p.W - 1;
  const int nslot = static_cast<int>(q_first + S - first);
  if (!dbg_ok(p.status, first >= 0 && first + nslot <= I && gq < p.total_quads)) {
    grid_dependency_wait();
    return;
  }

  grid_dependency_wait();  // every partial of the streaming kernel is written and visible
  const int chunk = p.red_chunk;
  const int per_quad = p.M * 64;  // floats per partial slot
  const uint32_t slot_bytes = static_cast<uint32_t>(per_quad) * 4u;
  const int stage_floats = chunk * per_quad;
  const float* buf = reinterpret_cast<const float*>(rsm);
  const uint32_t buf0 = smem_addr(rsm), bar0 = smem_addr(rsm + 2 * stage_floats * 4);
  const float* src = p.partials + first * per_quad;
  const int nchunks = div_up(nslot, chunk);
  uint64_t pol = 0;
  auto issue = [&](int ch) {
    const int ns = min(chunk, nslot - ch * chunk);
    const uint32_t bar = bar0 + 8 * (ch & 1);
    mbar_arrive_expect_tx(bar, ns * slot_bytes);
    bulk_g2s(buf0 + (ch & 1) * stage_floats * 4, src + static_cast<long long>(ch) * stage_floats, ns * slot_bytes,
             bar, pol);
  };
  if (threadIdx.x == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    fence_mbar_init();
    pol = l2_policy_evict_first();  // partials are read once
    issue(0);
    if (nchunks > 1) issue(1);
  }
  const int u = threadIdx.x, row = u >> 4, col = 4 * (u & 15);
  const bool active = row < p.M && col < kTileN * min(kQuadTiles, T - kQuadTiles * q);
  const long long i = static_cast<long long>(row) * m.N + kQuadTiles * kTileN * q + col;
  uint32_t r0 = 0u, r1 = 0u;  // the residual, loaded while the partials are in flight
  if (active) {
    r0 = residual2<NORM>(p, i);
    r1 = residual2<NORM>(p, i + 2);
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int ch = 0; ch < nchunks; ++ch) {
    if (threadIdx.x == 0) {
      const bool got = mbar_wait_bounded(bar0 + 8 * (ch & 1), (ch >> 1) & 1, p.wait_ns);
      if (!got) {
        // record the timeout and wait (bounded) for the other stage's copy
        atomicCAS(p.status, 0u, static_cast<unsigned>(W4G128_ERR_TIMEOUT));
        if (ch + 1 < nchunks) (void)mbar_wait_bounded(bar0 + 8 * ((ch + 1) & 1), ((ch + 1) >> 1) & 1, p.wait_ns);
      }
      ok = got;
    }
    __syncthreads();
    if (!ok) return;
    if (active) {
      const float* b = buf + (ch & 1) * stage_floats + row * 64 + col;
      const int ns = min(chunk, nslot - ch * chunk);
      for (int s = 0; s < ns; ++s) {
        const float4 v = *reinterpret_cast<const float4*>(b + s * per_quad);
        if (ch == 0 && s == 0) {
          acc = v;
        } else {
          acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
      }
    }
    __syncthreads();  // the stage is consumed before it is refilled
    if (threadIdx.x == 0 && ch + 2 < nchunks) {
      fence_proxy_async_smem();
      issue(ch + 2);
    }
  }
  if (active) {
    uint32_t* yo = reinterpret_cast<uint32_t*>(m.y + i);
    yo[0] = emit2<NORM>(acc.x, acc.y, r0);
    yo[1] = emit2<NORM>(acc.z, acc.w, r1);
  }
}

// Per streaming warp (calls with more quads than warps: most quads are owned
// by one warp, and a grid over quads would be mostly idle CTAs): one CTA per
// streaming warp w.  If the quad w's range starts in began in warp w - 1, w
// is the quad's second warp and its CTA folds the quad: the slots run from
// w - 1's last item (its prefix fold) to the quad's last segment.  With one
// matrix the CTA works out w's quad from the schedule; with several it reads
// w's record (no search of the matrix table).  Both happen before the wait.
constexpr int kRedBatch = 8;  // partial loads in flight per thread (register budget)

template <int MAXMAT, bool NORM>
__global__ void __launch_bounds__(kRedThreads) reduce_warps_kernel(const __grid_constant__ StreamParams<MAXMAT> p) {
  // as in reduce_quads_kernel: every CTA that folds waits for the streaming
  // grid, and so does the last
  grid_dependents_launch();
  const int w = blockIdx.x;
  const long long I = p.total_items;
  const long long it_a = I * w / p.W;
  bool split = false;
  int mi = 0, q = 0, s = 0;
  if constexpr (MAXMAT > 1) {
    __shared__ unsigned long long rec_s;
    if (threadIdx.x == 0) {
      unsigned long long r = 0ull;
      if (!wait_nonzero_bounded(p.recs + w, r, p.wait_ns))
        atomicCAS(p.status, 0u, static_cast<unsigned>(W4G128_ERR_TIMEOUT));
      rec_s = r;
    }
    __syncthreads();
    const unsigned long long rec = rec_s;
    split = (rec & kRecSplit) != 0;
    mi = static_cast<int>((rec >> 44) & 0x1FF);
    q = static_cast<int>((rec >> 20) & 0xFFFFFF);
    s = static_cast<int>(rec & 0xFFFFF);
  } else if (w > 0) {
    const int S = div_up(p.mats[0].K / kGroup, kSegGroups);
    q = static_cast<int>(it_a / S);
    s = static_cast<int>(it_a - static_cast<long long>(q) * S);
    split = s != 0 && it_a - s >= I * (w - 1) / p.W;
  }
  if (!split) {
    if (blockIdx.x + 1 == gridDim.x) grid_dependency_wait();
    return;
  }
  const MatParams& m = mat(p, mi);
  const int S = div_up(m.K / kGroup, kSegGroups);
  const int nslot = S - s + 1;
  if (!dbg_ok(p.status, it_a - 1 >= 0 && it_a - 1 + nslot <= I && mi < p.count)) {
    grid_dependency_wait();
    return;
  }
  const int cols = kTileN * min(kQuadTiles, m.N / kTileN - kQuadTiles * q);
  const int u = threadIdx.x, row = u >> 4, col = 4 * (u & 15);
  const bool active = row < p.M && col < cols;
  const long long i = static_cast<long long>(row) * m.N + kQuadTiles * kTileN * q + col;
  uint32_t r0 = 0u, r1 = 0u;  // the residual, loaded before the wait
  if (active) {
    r0 = residual2<NORM>(p, i);
    r1 = residual2<NORM>(p, i + 2);
  }
  uint16_t* y = m.y;
  grid_dependency_wait();  // every partial of the streaming kernel is written and visible
  if (!active) return;
  const int per_quad = p.M * 64;  // floats per partial slot
  const float4* part = reinterpret_cast<const float4*>(p.partials + (it_a - 1) * per_quad + row * 64 + col);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < nslot; s0 += kRedBatch) {  // kRedBatch slots in flight, then fold in order
    float4 v[kRedBatch];
#pragma unroll
    for (int k = 0; k < kRedBatch; ++k)
      v[k] = (s0 + k < nslot) ? __ldcg(part + static_cast<long long>(s0 + k) * (per_quad / 4))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kRedBatch; ++k) {
      if (s0 + k < nslot) {
        if (s0 + k == 0) {
          acc = v[k];
        } else {
          acc.x += v[k].x; acc.y += v[k].y; acc.z += v[k].z; acc.w += v[k].w;
        }
      }
    }
  }
  uint32_t* yo = reinterpret_cast<uint32_t*>(y + i);
  yo[0] = emit2<NORM>(acc.x, acc.y, r0);
  yo[1] = emit2<NORM>(acc.z, acc.w, r1);
}

// ----------------------------------------------------------------- RMS norm kernel

// The residual add + RMS norm call ends in this kernel, launched behind the
// call's last kernel (programmatic dependent launch): every h is written and
// visible once it has waited.  One CTA per (row m, slice of kNormSlice 8-column
// chunks) normalises its slice of row m:
//   out[m][n] = bf16( fl(fl(h[m][n] r_m) gamma[n]) ),
//   r_m = 1 / sqrt( fl(S_m / N) + eps )   (one correctly rounded fp32 op each),
// with S_m = sum_n h[m][n]^2 summed in an order fixed by N alone: the row is
// cut into 8-column chunks dealt round robin to the 256 threads (chunk j to
// thread j mod 256); a thread folds the squares of its chunks' columns in
// column order with fp32 FMAs; a xor butterfly adds each warp's 32 sums; the
// 8 warp sums are added as a balanced tree.  Every CTA of a row computes the
// same S_m from the whole row (a few KB from L2) and keeps the chunks of its
// own slice in shared memory for the output pass.
constexpr int kNormThreads = 256;
constexpr int kNormSlice = 128;  // chunks (1024 columns) per CTA

__device__ __forceinline__ float sq_word(uint32_t v, float acc) {
  acc = fmaf(bf16_lo(v), bf16_lo(v), acc);
  return fmaf(bf16_hi(v), bf16_hi(v), acc);
}

// out word = bf16 pair of (h * r) * g, element by element
__device__ __forceinline__ uint32_t norm_word(uint32_t h, uint32_t g, float r) {
  const float2 v = fmul2(fmul2(make_float2(bf16_lo(h), bf16_hi(h)), make_float2(r, r)),
                         make_float2(bf16_lo(g), bf16_hi(g)));
  uint32_t o;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o) : "f"(v.y), "f"(v.x));  // (hi, lo)
  return o;
}

// 8 columns (4 words) at a: one 16-byte access when `vec`, else four 4-byte
// ones (rows need only 4-byte alignment)
__device__ __forceinline__ uint4 load_chunk(const uint32_t* a, bool vec) {
  if (vec) return __ldcg(reinterpret_cast<const uint4*>(a));
  return make_uint4(__ldcg(a), __ldcg(a + 1), __ldcg(a + 2), __ldcg(a + 3));
}

__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const __grid_constant__ StreamParams<1> p) {
  __shared__ uint4 mine[kNormSlice];
  __shared__ float wsum[kNormThreads / 32];
  __shared__ float r_row;
  // The next call's prep kernel may launch now; it waits for this grid.
  grid_dependents_launch();
  grid_dependency_wait();
  if ((*reinterpret_cast<volatile unsigned*>(p.status) & 0xFFu) != 0u) return;  // the product failed: out left unwritten
  const MatParams& m = p.mats[0];
  const int row = blockIdx.y, j0 = blockIdx.x * kNormSlice, t = threadIdx.x;
  const int npairs = m.N >> 1, nchunk = npairs >> 2;
  const uint32_t* h = reinterpret_cast<const uint32_t*>(m.y) + static_cast<long long>(row) * npairs;
  const uint32_t* gam = reinterpret_cast<const uint32_t*>(p.gamma);
  uint32_t* out = reinterpret_cast<uint32_t*>(p.nout) + static_cast<long long>(row) * npairs;
  // rows start 32-byte aligned relative to the base (N % 16 == 0): one test per array
  const bool hvec = (reinterpret_cast<uintptr_t>(m.y) & 15u) == 0u;
  const bool gvec = (reinterpret_cast<uintptr_t>(p.gamma) & 15u) == 0u;
  const bool ovec = (reinterpret_cast<uintptr_t>(p.nout) & 15u) == 0u;
  float acc = 0.f;
#pragma unroll 4
  for (int j = t; j < nchunk; j += kNormThreads) {
    const uint4 v = load_chunk(h + 4 * j, hvec);
    acc = sq_word(v.w, sq_word(v.z, sq_word(v.y, sq_word(v.x, acc))));
    if (j >= j0 && j < j0 + kNormSlice) mine[j - j0] = v;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((t & 31) == 0) wsum[t >> 5] = acc;
  __syncthreads();
  if (t == 0) {
    const float S = ((wsum[0] + wsum[1]) + (wsum[2] + wsum[3])) + ((wsum[4] + wsum[5]) + (wsum[6] + wsum[7]));
    r_row = __frsqrt_rn(__fadd_rn(__fdiv_rn(S, static_cast<float>(m.N)), p.eps));
  }
  __syncthreads();
  const int j = j0 + t;
  if (t < kNormSlice && j < nchunk) {
    const uint4 v = mine[t], g = load_chunk(gam + 4 * j, gvec);
    const float r = r_row;
    const uint4 o = make_uint4(norm_word(v.x, g.x, r), norm_word(v.y, g.y, r), norm_word(v.z, g.z, r),
                               norm_word(v.w, g.w, r));
    if (ovec) {
      *reinterpret_cast<uint4*>(out + 4 * j) = o;
    } else {
      out[4 * j] = o.x;
      out[4 * j + 1] = o.y;
      out[4 * j + 2] = o.z;
      out[4 * j + 3] = o.w;
    }
  }
}

// ----------------------------------------------------------------- host planning

struct DeviceInfo {
  int sms = 0;
  int occ[4] = {0, 0, 0, 0};        // CTAs per SM per mode
  int red_occ[kMaxRows + 1] = {};   // per-quad reduce CTAs per SM per M
  int red_occ_deep[kMaxRows + 1] = {};  // the same at kRedChunkDeep slots per copy
  int pair_clusters = 0;            // clusters of two local M = 1 CTAs resident at once
  bool ok = false;
};

std::mutex g_mu;
DeviceInfo g_dev[64];
std::atomic<bool> g_dev_init[64];  // set once g_dev[i] is filled (released under g_mu)

void setup_local() {
  cudaFuncSetAttribute(fold1_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFoldSmem);
  cudaFuncSetAttribute(fold1_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFoldSmem);
  cudaFuncSetAttribute(fold1_kernel<kFewMatrices, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFoldSmem);
  cudaFuncSetAttribute(fold1_kernel<W4G128_MAX_MATRICES, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       kFoldSmem);
  cudaFuncSetAttribute(stream1_local_kernel<1, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLocalDyn);
  cudaFuncSetAttribute(stream1_local_kernel<1, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLocalDyn);
  cudaFuncSetAttribute(stream1_local_kernel<1, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLocalDyn);
  cudaFuncSetAttribute(stream1_local_kernel<1, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLocalDyn);
  cudaFuncSetAttribute(stream1_local_kernel<kFewMatrices, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       kLocalDyn);
  cudaFuncSetAttribute(stream1_local_kernel<W4G128_MAX_MATRICES, false, false>,
                       cudaFuncAttributeMaxDynamicSharedMemorySize, kLocalDyn);
}

template <int MODE>
void setup_mode(DeviceInfo& d) {
  const int smem = smem_bytes<MODE>();
  cudaFuncSetAttribute(stream_kernel<MODE, 1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaFuncSetAttribute(stream_kernel<MODE, 1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if constexpr (MODE == kMMA) {
    cudaFuncSetAttribute(stream_kernel<MODE, 1, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(stream_kernel<MODE, 1, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  }
  cudaFuncSetAttribute(stream_kernel<MODE, kFewMatrices, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaFuncSetAttribute(stream_kernel<MODE, W4G128_MAX_MATRICES, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       smem);
  cudaFuncSetAttribute(reduce_quads_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRedSmem);
  cudaFuncSetAttribute(reduce_quads_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRedSmem);
  cudaFuncSetAttribute(reduce_quads_kernel<kFewMatrices, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       kRedSmem);
  cudaFuncSetAttribute(reduce_quads_kernel<W4G128_MAX_MATRICES, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       kRedSmem);
  int occ1 = 0, occ2 = 0, occ3 = 0;
  constexpr int threads = cta_warps_max<MODE>() * 32;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ1, stream_kernel<MODE, 1, false>, threads, smem);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ2, stream_kernel<MODE, W4G128_MAX_MATRICES, false>, threads,
                                                smem);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ3, stream_kernel<MODE, 1, true>, threads, smem);
  occ2 = std::min(occ2, occ3);
  const int occ = std::min(occ1, occ2);
  d.occ[MODE] = occ > 0 ? occ : 1;
}

const DeviceInfo* device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return nullptr;
  }
  if (g_dev_init[dev].load(std::memory_order_acquire)) return &g_dev[dev];  // the per-call path
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_dev_init[dev].load(std::memory_order_relaxed)) {
    DeviceInfo d;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    d.ok = (major == 10 && minor == 3);
    if (d.ok) {
      setup_mode<kMMA>(d);
      setup_mode<kMMA1>(d);
      setup_mode<kMMA16>(d);
      setup_local();
      {
        // how many two-CTA clusters of the local kernel (both forms paired
        // quads use) fit on the device at once
        cudaLaunchAttribute ca[1];
        ca[0].id = cudaLaunchAttributeClusterDimension;
        ca[0].val.clusterDim.x = 2;
        ca[0].val.clusterDim.y = 1;
        ca[0].val.clusterDim.z = 1;
        cudaLaunchConfig_t cc = {};
        cc.gridDim = dim3(2);
        cc.blockDim = dim3(kWideWarps * 32);
        cc.dynamicSmemBytes = kLocalDyn;
        cc.attrs = ca;
        cc.numAttrs = 1;
        int n = 0, n16 = 0;
        if (cudaOccupancyMaxActiveClusters(&n, stream1_local_kernel<1, false, true>, &cc) != cudaSuccess) {
          cudaGetLastError();
          n = 0;
        }
        cc.blockDim = dim3(kNW * 32);
        if (cudaOccupancyMaxActiveClusters(&n16, stream1_local_kernel<1, false, false>, &cc) != cudaSuccess) {
          cudaGetLastError();
          n16 = 0;
        }
        d.pair_clusters = std::min(n, n16);
      }
      for (int M = 2; M <= kMaxRows; ++M) {
        int n = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, reduce_quads_kernel<W4G128_MAX_MATRICES, false>,
                                                      red_threads(M), red_smem(M));
        d.red_occ[M] = n > 0 ? n : 1;
        n = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, reduce_quads_kernel<W4G128_MAX_MATRICES, false>,
                                                      red_threads(M), red_smem(M, kRedChunkDeep));
        d.red_occ_deep[M] = n;
      }
      if (cudaGetLastError() != cudaSuccess) d.ok = false;
    }
    g_dev[dev] = d;
    g_dev_init[dev].store(true, std::memory_order_release);
  }
  return &g_dev[dev];
}

// Drops the current device's cached set-up (kernel attributes, occupancy).
void forget_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  g_dev_init[dev].store(false, std::memory_order_release);
}

struct Plan {
  int mode = 0, rows = 1, pkg = 0, depth = 2;
  bool per_warp_reduce = false;
  int red_chunk = kRedChunk;  // per-quad fold: slots per bulk copy
  bool red_reverse = false;   // per-quad fold: deepest (last) quads first
  bool local = false;   // M = 1 with CTA-local packages (when x is 16-byte aligned)
  int local_depth = 2;  // ring slots per warp of a local call
  int local_pkg_off = 0, local_part_off = 0;
  long long items = 0;
  int W = 0, grid = 0, cta_warps = kNW, total_quads = 0, total_groups = 0, max_groups = 0;
  size_t off_tickets = 0, off_recs = 0, off_xpkg = 0, off_partials = 0, bytes = 0;
  std::vector<long long> item_begin, xpkg_off;
  std::vector<int> quad_begin, g_begin;
  std::vector<long long> cta_begin;  // local calls of up to kFewMatrices matrices: the CTAs' first items
  bool whole_quads = false;          // M = 1, one matrix: one CTA per quad, no boundary fold
  bool pair_quads = false;           // M = 1, one matrix: two CTAs (a cluster) per quad, no boundary fold
  // The balanced split (W <= items: every warp has an item), which the
  // package-kernel path takes when the local kernel cannot (x not 16-byte
  // aligned): the paired quads give a warp no item when S is odd, and that
  // path's ticket count takes every warp between a quad's owners to hold
  // some of it.
  int gen_grid = 0, gen_cta_warps = 0, gen_W = 0;
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool make_plan(const HostMatrix* mats, int count, int M, const DeviceInfo& dev, Plan& pl) {
  pl = Plan();  // cached plans are reused: start from the defaults
  pl.mode = (M > 8) ? kMMA16 : (M > 1) ? kMMA : kMMA1;
  pl.rows = M;
  pl.pkg = (pl.mode == kMMA16) ? Pkg<kMMA16>::kBytes : (pl.mode == kMMA) ? Pkg<kMMA>::kBytes : Pkg<kMMA1>::kBytes;
  pl.item_begin.resize(count);
  pl.quad_begin.resize(count);
  pl.g_begin.resize(count);
  pl.xpkg_off.resize(count);
  long long items = 0, xbytes = 0, quads = 0, groups = 0;
  for (int i = 0; i < count; ++i) {
    const int seg = kSegGroups;
    const int G = mats[i].K / kGroup, S = div_up(G, seg), NQ = div_up(mats[i].N, kTileN * kQuadTiles);
    pl.item_begin[i] = items;
    pl.quad_begin[i] = static_cast<int>(quads);
    pl.g_begin[i] = static_cast<int>(groups);
    pl.xpkg_off[i] = xbytes;
    items += static_cast<long long>(NQ) * S;
    quads += NQ;
    groups += G;
    pl.max_groups = std::max(pl.max_groups, G);
    xbytes += static_cast<long long>(G) * pl.pkg;
    if (quads > (1 << 24) || groups > 0x7FFFFFFF) return false;  // quad indices stay well inside int
  }
  pl.items = items;
  pl.total_quads = static_cast<int>(quads);
  pl.total_groups = static_cast<int>(groups);
  const int nw = (pl.mode == kMMA16) ? cta_warps_max<kMMA16>() : kNW;
  const long long max_warps = static_cast<long long>(dev.sms) * dev.occ[pl.mode] * nw;
  // Warps: as many as the grid holds, but with a whole number of items each
  // when a warp gets only a few: the warps of a call finish together instead
  // of some streaming one item more than the rest (2720 items on 2432 warps
  // would give most warps one item and some two).  The summation order
  // depends on the segments alone, so the schedule changes no bit.
  const long long per = (items + max_warps - 1) / max_warps;  // items per warp, at least
  pl.W = static_cast<int>(per < 4 ? (items + per - 1) / per : std::min<long long>(items, max_warps));
  // Spread the warps over every SM: a call with fewer items than the grid
  // holds warps gets smaller CTAs rather than fewer SMs.
  pl.cta_warps = std::min(nw, div_up(pl.W, dev.sms));
  pl.grid = div_up(pl.W, pl.cta_warps);
  pl.gen_grid = pl.grid;
  pl.gen_cta_warps = pl.cta_warps;
  pl.gen_W = pl.W;
  pl.depth = (pl.mode == kMMA1) ? ring_depth<kMMA1>() : ring_depth<kMMA>();
  // M >= 2: fold per quad unless that grid is larger than one streaming warp
  // each and than one wave of resident reduce CTAs
  pl.per_warp_reduce = M >= 2 && pl.total_quads > pl.W &&
                       static_cast<long long>(pl.total_quads) > static_cast<long long>(dev.red_occ[M]) * dev.sms;
  // Per-quad fold: quads deeper than kRedChunk segments are copied
  // kRedChunkDeep slots at a time when every fold CTA still fits one wave at
  // that stage size (fewer dependent copy rounds; measured 17408x5120 at
  // M = 8 18.8 -> 17.4 us, 6144x5120 9.8 -> 9.0 us); a call whose last matrix
  // is its deepest (a layer: down) folds from the last quad back, so the
  // longest folds start first (layer step M = 8 43.0 -> 42.5 us, M = 16
  // 69.8 -> 68.7 us).
  if (M >= 2 && !pl.per_warp_reduce) {
    int smax = 0, slast = 0;
    for (int i = 0; i < count; ++i) {
      const int S = div_up(mats[i].K / kGroup, kSegGroups);
      smax = std::max(smax, S);
      slast = S;
    }
    if (M <= 8 && smax > kRedChunk &&
        static_cast<long long>(pl.total_quads) <= static_cast<long long>(dev.red_occ_deep[M]) * dev.sms)
      pl.red_chunk = kRedChunkDeep;
    pl.red_reverse = count > 1 && slast == smax;
  }

  // Local calls of up to kFewMatrices matrices take the CTAs' item ranges
  // from a table in the kernel parameters (the balanced split), which each
  // CTA reads before its dependency wait instead of deriving it.
  const bool cta_table = pl.mode == kMMA1 && count <= kFewMatrices;
  // A single matrix of between sms / 4 and sms quads of at most
  // kWholeQuadSegs segments runs one CTA per quad, one warp per segment: no
  // quad straddles two CTAs, so the boundary fold kernel is not launched
  // (measured: 4096^2 6.8 -> 6.5 us, 5120x6144 8.8 -> 8.1 us; at 12 segments,
  // 6144x5120, the larger per-SM share cancels the gain).
  constexpr int kWholeQuadSegs = 10;
  if (cta_table && count == 1) {
    const int S1 = div_up(mats[0].K / kGroup, kSegGroups);
    const int NQ1 = div_up(mats[0].N, kTileN * kQuadTiles);
    if (S1 <= kWholeQuadSegs && NQ1 <= dev.sms && 4 * NQ1 >= dev.sms) {
      pl.grid = NQ1;
      pl.cta_warps = S1;
      pl.W = NQ1 * S1;
      pl.whole_quads = true;
    }
    // Deeper quads (up to two CTAs' worth of warps), when clusters of two
    // CTAs fit once per quad: quad q's segments are split between CTAs 2q and
    // 2q + 1, which fold through the first one's shared memory, so no quad
    // needs the boundary fold kernel.  The pairs leave sms - 2 NQ SMs idle
    // that the balanced split would use; they are taken while the extra
    // bytes each streaming SM then pulls, ceil(S / 2) items x (1 - 2 NQ /
    // sms), stay within 4 items (measured, us, pairs against the balanced
    // split with its fold kernel: 8192x4096 8.37 / 8.94, 11392x4080 9.48 /
    // 10.73, 16384x4096 11.45 / 12.40, 10240x3072 8.54 / 8.76, 5632x2432
    // 6.77 / 6.84; 16384x2432, 16 items x 1/2, 10.15 / 8.86).  Not for quads
    // one CTA holds: there each warp's chunks are a latency-bound sequence
    // whatever the CTAs per SM, and pairs only add the cluster barrier
    // (4096^2 6.58 against 6.07 us with one CTA per quad).
    else if (S1 > kWholeQuadSegs && S1 <= 2 * kNW && NQ1 <= dev.pair_clusters && 4 * NQ1 >= dev.sms &&
             div_up(S1, 2) * (dev.sms - 2 * NQ1) <= 4 * dev.sms) {
      pl.grid = 2 * NQ1;
      pl.cta_warps = div_up(S1, 2);
      pl.W = pl.grid * pl.cta_warps;
      pl.whole_quads = true;
      pl.pair_quads = true;
    }
  }
  if (pl.pair_quads) {
    const int S1 = div_up(mats[0].K / kGroup, kSegGroups);
    pl.cta_begin.resize(pl.grid + 1);
    for (int q = 0; q < pl.grid / 2; ++q) {
      pl.cta_begin[2 * q] = static_cast<long long>(q) * S1;
      pl.cta_begin[2 * q + 1] = static_cast<long long>(q) * S1 + div_up(S1, 2);
    }
    pl.cta_begin[pl.grid] = items;
  } else if (cta_table && pl.grid <= kMaxLocalCtas) {
    pl.cta_begin.resize(pl.grid + 1);
    for (int c = 0; c <= pl.grid; ++c)
      pl.cta_begin[c] = items * std::min<long long>(static_cast<long long>(c) * pl.cta_warps, pl.W) / pl.W;
  }

  // M = 1: can every CTA hold its packages and partial slots in shared memory?
  if (pl.mode == kMMA1) {
    struct HostMats {
      const Plan& pl;
      const HostMatrix* m;
      long long begin(int i) const { return pl.item_begin[i]; }
      int K(int i) const { return m[i].K; }
      int N(int i) const { return m[i].N; }
    } at{pl, mats};
    int pmax = 0;
    long long smax = 0;
    bool ok = true;
    if (cta_table && pl.cta_begin.empty()) ok = false;  // more CTAs than the table holds
    for (int c = 0; c < pl.grid && ok; ++c) {
      const long long A = cta_table ? pl.cta_begin[c] : items * (static_cast<long long>(c) * pl.cta_warps) / pl.W;
      const long long B = cta_table ? pl.cta_begin[c + 1]
                                    : items * std::min((c + 1) * pl.cta_warps, pl.W) / pl.W;
      LocalEntry t[kLocalMaxEntries];
      int np = 0;
      if (local_table(A, B, count, at, t, np) < 0) ok = false;
      pmax = std::max(pmax, np);
      smax = std::max(smax, B - A);
    }
    if (pl.pair_quads) smax = std::max<long long>(smax, div_up(mats[0].K / kGroup, kSegGroups));  // the leader
    ok = ok && static_cast<long long>(pmax) * kPkg1 + smax * 64 * 4 <= kLocalSpace;
    pl.local = ok;
    pl.local_depth = std::min(8, kLocalSlots / pl.cta_warps);
    pl.local_pkg_off = kLocalBarBytes + kLocalRing;
    pl.local_part_off = pl.local_pkg_off + pmax * kPkg1;
  }

  pl.off_tickets = 256;  // after the status word
  pl.off_recs = align_up(pl.off_tickets + sizeof(unsigned) * static_cast<size_t>(quads), 256);
  pl.off_xpkg = align_up(pl.off_recs + sizeof(unsigned long long) * static_cast<size_t>(pl.W), 256);
  pl.off_partials = align_up(pl.off_xpkg + static_cast<size_t>(xbytes), 256);
  pl.bytes = align_up(pl.off_partials + sizeof(float) * static_cast<size_t>(items) * pl.rows * 64, 256);
  return true;
}

template <int MAXMAT>
void fill_params(StreamParams<MAXMAT>& sp, const HostMatrix* mats, int count, int M, const Plan& pl,
                 const NormArgs* norm, void* ws) {
  auto* base = static_cast<uint8_t*>(ws);
  sp.total_items = pl.items;
  sp.partials = reinterpret_cast<float*>(base + pl.off_partials);
  sp.tickets = reinterpret_cast<unsigned*>(base + pl.off_tickets);
  sp.recs = reinterpret_cast<unsigned long long*>(base + pl.off_recs);
  sp.status = reinterpret_cast<unsigned*>(base);
  sp.residual = norm ? norm->residual : nullptr;
  sp.gamma = norm ? norm->gamma : nullptr;
  sp.nout = norm ? norm->out : nullptr;
  sp.eps = norm ? norm->eps : 0.f;
  sp.count = count;
  sp.M = M;
  sp.W = pl.W;
  sp.per_warp_reduce = pl.per_warp_reduce ? 1 : 0;
  sp.red_chunk = pl.red_chunk;
  sp.red_reverse = pl.red_reverse ? 1 : 0;
  sp.depth = pl.depth;
  sp.wait_ns = kDefaultWaitNs;
  sp.cta_warps = pl.cta_warps;
  sp.local_pkg_off = pl.local_pkg_off;
  sp.local_part_off = pl.local_part_off;
  sp.pair = 0;  // set by the local launch
  if constexpr (MAXMAT <= kFewMatrices) {
    const int nb = std::min(static_cast<int>(pl.cta_begin.size()), kMaxLocalCtas + 1);
    for (int c = 0; c < nb; ++c) sp.cta_begin[c] = pl.cta_begin[c];
  }
  sp.total_quads = pl.total_quads;
  sp.total_groups = pl.total_groups;
  for (int i = 0; i < count; ++i) {
    MatParams& m = sp.mats[i];
    m.packed = static_cast<const uint8_t*>(mats[i].packed);
    m.xpkg = base + pl.off_xpkg + pl.xpkg_off[i];
    m.x = mats[i].x;
    m.y = mats[i].y;
    m.item_begin = pl.item_begin[i];
    m.K = mats[i].K;
    m.N = mats[i].N;
    m.quad_begin = pl.quad_begin[i];
    m.g_begin = pl.g_begin[i];
  }
}

// M = 1 with CTA-local packages: the streaming kernel (a programmatic
// dependent of whatever precedes it), the boundary fold behind it when CTA
// boundaries can split quads, and the norm behind that.
template <int MAXMAT, bool NORM, bool WIDE>
int launch_local(const StreamParams<MAXMAT>& sp, int grid, int cta_warps, bool boundary_fold, cudaStream_t stream) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;  // paired quads: clusters of two CTAs
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = sp.pair ? 2 : 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(cta_warps * 32);
  cfg.dynamicSmemBytes = kLocalDyn;
  if (cudaLaunchKernelEx(&cfg, stream1_local_kernel<MAXMAT, NORM, WIDE>, sp) != cudaSuccess) {
    cudaGetLastError();
    return W4G128_ERR_CUDA;
  }
  cfg.numAttrs = 1;
  if (grid > 1 && boundary_fold) {
    cfg.gridDim = dim3(grid - 1);
    cfg.blockDim = dim3(32);
    cfg.dynamicSmemBytes = kFoldSmem;
    if (cudaLaunchKernelEx(&cfg, fold1_kernel<MAXMAT, NORM>, sp) != cudaSuccess) {
      cudaGetLastError();
      return W4G128_ERR_CUDA;
    }
  }
  if constexpr (NORM) {
    const int nchunk = sp.mats[0].N / 8;
    cfg.gridDim = dim3(static_cast<unsigned>(div_up(nchunk, kNormSlice)), static_cast<unsigned>(sp.M));
    cfg.blockDim = dim3(kNormThreads);
    cfg.dynamicSmemBytes = 0;
    if (cudaLaunchKernelEx(&cfg, rmsnorm_kernel, sp) != cudaSuccess) {
      cudaGetLastError();
      return W4G128_ERR_CUDA;
    }
  }
  return W4G128_OK;
}

template <int MODE, int MAXMAT, bool NORM>
int launch_mode(const StreamParams<MAXMAT>& sp, int grid, int cta_warps, int max_groups, cudaStream_t stream) {
  // Every kernel of the call is a programmatic dependent launch: the prep
  // kernel behind whatever precedes it in the stream (it waits for that to
  // finish before touching anything), the streaming kernel behind the prep
  // kernel (its weight copies start before it waits), the reduce kernel
  // behind the streaming kernel.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.dynamicSmemBytes = 0;
  cudaError_t e;
  cfg.gridDim = dim3(static_cast<unsigned>(std::min(div_up(max_groups, 8), 4096)), static_cast<unsigned>(sp.count));
  if constexpr (multi_row<MODE>()) {
    cfg.blockDim = dim3(256);
    e = cudaLaunchKernelEx(&cfg, prep_kernel<MODE, MAXMAT>, sp);
  } else {
    cfg.blockDim = dim3(32);
    e = cudaLaunchKernelEx(&cfg, prep1_kernel<MODE, MAXMAT>, sp);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return W4G128_ERR_CUDA;
  }
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(cta_warps * 32);
  // the full CTA's shared memory even for smaller CTAs: one CTA per SM, so a
  // call with few warps still spreads over every SM instead of packing two
  // CTAs onto one
  cfg.dynamicSmemBytes = smem_bytes<MODE>();
  bool wide = false;
  if constexpr (MODE == kMMA && MAXMAT == 1) wide = cta_warps <= kWideWarps;
  cudaError_t es;
  if constexpr (MODE == kMMA && MAXMAT == 1) {
    es = wide ? cudaLaunchKernelEx(&cfg, stream_kernel<MODE, 1, NORM, true>, sp)
              : cudaLaunchKernelEx(&cfg, stream_kernel<MODE, 1, NORM>, sp);
  } else {
    es = cudaLaunchKernelEx(&cfg, stream_kernel<MODE, MAXMAT, NORM>, sp);
  }
  if (es != cudaSuccess) {
    cudaGetLastError();
    return W4G128_ERR_CUDA;
  }
  if (multi_row<MODE>()) {  // M >= 2: the split quads are folded by the reduce kernel
    cudaError_t er;
    cfg.blockDim = dim3(red_threads(sp.M));
    if (sp.per_warp_reduce) {
      cfg.gridDim = dim3(static_cast<unsigned>(sp.W));  // one CTA per streaming warp
      cfg.dynamicSmemBytes = 0;
      er = cudaLaunchKernelEx(&cfg, reduce_warps_kernel<MAXMAT, NORM>, sp);
    } else {
      cfg.gridDim = dim3(static_cast<unsigned>(sp.total_quads));  // one CTA per quad
      cfg.dynamicSmemBytes = red_smem(sp.M, sp.red_chunk);
      er = cudaLaunchKernelEx(&cfg, reduce_quads_kernel<MAXMAT, NORM>, sp);
    }
    if (er != cudaSuccess) {
      cudaGetLastError();
      return W4G128_ERR_CUDA;
    }
  }
  if constexpr (NORM) {
    static_assert(MAXMAT == 1, "the residual add + RMS norm call streams one matrix");
    const int nchunk = sp.mats[0].N / 8;
    cfg.gridDim = dim3(static_cast<unsigned>(div_up(nchunk, kNormSlice)), static_cast<unsigned>(sp.M));
    cfg.blockDim = dim3(kNormThreads);
    cfg.dynamicSmemBytes = 0;
    if (cudaLaunchKernelEx(&cfg, rmsnorm_kernel, sp) != cudaSuccess) {
      cudaGetLastError();
      return W4G128_ERR_CUDA;
    }
  }
  return W4G128_OK;
}

// Local calls stage x with bulk copies, which need 16-byte aligned sources.
bool x_aligned(const HostMatrix* mats, int count) {
  for (int i = 0; i < count; ++i)
    if ((reinterpret_cast<uintptr_t>(mats[i].x) & 15u) != 0u) return false;
  return true;
}

template <int MAXMAT>
int launch_with(const HostMatrix* mats, int count, int M, const Plan& pl, const NormArgs* norm, void* ws,
                cudaStream_t stream) {
  static thread_local StreamParams<MAXMAT> sp;  // large for MAXMAT = 512: keep it off the stack
  fill_params(sp, mats, count, M, pl, norm, ws);
  if (pl.local && x_aligned(mats, count)) {
    sp.depth = pl.local_depth;
    sp.pair = pl.pair_quads ? 1 : 0;
    if constexpr (MAXMAT == 1) {
      if (pl.cta_warps <= kWideWarps) {
        if (norm != nullptr) return launch_local<1, true, true>(sp, pl.grid, pl.cta_warps, !pl.whole_quads, stream);
        return launch_local<1, false, true>(sp, pl.grid, pl.cta_warps, !pl.whole_quads, stream);
      }
      if (norm != nullptr) return launch_local<1, true, false>(sp, pl.grid, pl.cta_warps, !pl.whole_quads, stream);
    }
    return launch_local<MAXMAT, false, false>(sp, pl.grid, pl.cta_warps, !pl.whole_quads, stream);
  }
  // the package-kernel path, over the balanced split
  sp.W = pl.gen_W;
  sp.cta_warps = pl.gen_cta_warps;
  const int grid = pl.gen_grid, cw = pl.gen_cta_warps;
  if constexpr (MAXMAT == 1) {
    if (norm != nullptr) {
      if (pl.mode == kMMA16) return launch_mode<kMMA16, 1, true>(sp, grid, cw, pl.max_groups, stream);
      if (pl.mode == kMMA) return launch_mode<kMMA, 1, true>(sp, grid, cw, pl.max_groups, stream);
      return launch_mode<kMMA1, 1, true>(sp, grid, cw, pl.max_groups, stream);
    }
  }
  if (pl.mode == kMMA16) return launch_mode<kMMA16, MAXMAT, false>(sp, grid, cw, pl.max_groups, stream);
  if (pl.mode == kMMA) return launch_mode<kMMA, MAXMAT, false>(sp, grid, cw, pl.max_groups, stream);
  return launch_mode<kMMA1, MAXMAT, false>(sp, grid, cw, pl.max_groups, stream);
}

// The last few plans of this host thread, keyed by device, M and the list of
// shapes: a decode loop repeats the same calls, and a plan (the schedule, the
// workspace layout, the per-CTA check of the local mode) depends on nothing
// else.
struct PlanCache {
  static constexpr int kEntries = 8;
  struct Entry {
    int dev = -1, M = 0;
    std::vector<int> shapes;  // K0, N0, K1, N1, ...
    Plan plan;
  } e[kEntries];
  int next = 0;
};

const Plan* cached_plan(const HostMatrix* mats, int count, int M, const DeviceInfo& info) {
  static thread_local PlanCache cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  for (auto& en : cache.e) {
    if (en.dev != dev || en.M != M || static_cast<int>(en.shapes.size()) != 2 * count) continue;
    bool same = true;
    for (int i = 0; i < count && same; ++i) same = en.shapes[2 * i] == mats[i].K && en.shapes[2 * i + 1] == mats[i].N;
    if (same) return &en.plan;
  }
  auto& en = cache.e[cache.next];
  cache.next = (cache.next + 1) % PlanCache::kEntries;
  en.dev = -1;
  if (!make_plan(mats, count, M, info, en.plan)) return nullptr;
  en.shapes.resize(2 * count);
  for (int i = 0; i < count; ++i) {
    en.shapes[2 * i] = mats[i].K;
    en.shapes[2 * i + 1] = mats[i].N;
  }
  en.dev = dev;
  en.M = M;
  return &en.plan;
}

}  // namespace

bool device_is_sm103() {
  const DeviceInfo* d = device_info();
  return d != nullptr && d->ok;
}

size_t stream_workspace_bytes(const HostMatrix* mats, int count, int M) {
  const DeviceInfo* d = device_info();
  if (d == nullptr || !d->ok) return 0;
  const Plan* pl = cached_plan(mats, count, M, *d);
  return pl == nullptr ? 0 : pl->bytes;
}

int launch_stream(const HostMatrix* mats, int count, int M, const NormArgs* norm, void* ws,
                  size_t ws_bytes, cudaStream_t stream) {
  const DeviceInfo* d = device_info();
  if (d == nullptr || !d->ok) return W4G128_ERR_DEVICE;
  const Plan* cached = cached_plan(mats, count, M, *d);
  if (cached == nullptr) return W4G128_ERR_SHAPE;
  const Plan& pl = *cached;
  if (ws_bytes < pl.bytes) return W4G128_ERR_WORKSPACE;
  if (norm != nullptr && count != 1) return W4G128_ERR_INVALID_ARG;
  int rc;
  if (count == 1) rc = launch_with<1>(mats, count, M, pl, norm, ws, stream);
  else if (count <= kFewMatrices) rc = launch_with<kFewMatrices>(mats, count, M, pl, norm, ws, stream);
  else rc = launch_with<W4G128_MAX_MATRICES>(mats, count, M, pl, norm, ws, stream);
  // A failed launch may mean the context was reset since the kernels'
  // attributes were set: the next call sets them up again.
  if (rc == W4G128_ERR_CUDA) forget_device();
  return rc;
}

int describe_schedule(const HostMatrix* mats, int count, int M, long long* out, int n) {
  const DeviceInfo* d = device_info();
  if (d == nullptr || !d->ok) return W4G128_ERR_DEVICE;
  const Plan* cached = cached_plan(mats, count, M, *d);
  if (cached == nullptr) return W4G128_ERR_SHAPE;
  const Plan& pl = *cached;
  bool xa = true;
  for (int i = 0; i < count; ++i)
    if (mats[i].x != nullptr && (reinterpret_cast<uintptr_t>(mats[i].x) & 15u) != 0u) xa = false;
  const bool local = pl.local && xa;
  long long v[8];
  v[0] = local ? 1 : 0;
  v[1] = local ? pl.grid : pl.gen_grid;
  v[2] = local ? pl.cta_warps : pl.gen_cta_warps;
  if (local) v[3] = (pl.grid > 1 && !pl.whole_quads) ? 1 : 0;
  else if (M == 1) v[3] = 0;  // the package-kernel path at M = 1 folds split quads inside the stream
  else v[3] = pl.per_warp_reduce ? 3 : 2;
  v[4] = (local && pl.pair_quads) ? 1 : 0;
  v[5] = local ? pl.local_depth : pl.depth;
  v[6] = static_cast<long long>(pl.bytes);
  v[7] = pl.items;
  for (int i = 0; i < n && i < 8; ++i) out[i] = v[i];
  return W4G128_OK;
}

int read_workspace_status(const void* ws, int* status_out, cudaStream_t stream) {
  unsigned v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return W4G128_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return W4G128_ERR_CUDA;
  *status_out = static_cast<int>(v & 0xFFu);  // the code byte (local calls tag the rest)
  return W4G128_OK;
}

}  // namespace w4g128
