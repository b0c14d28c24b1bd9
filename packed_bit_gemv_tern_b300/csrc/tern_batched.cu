// tern_batched.cu -- one persistent launch for a batch of independent ternary
// products: M = 1 GEMVs, small-M GEMMs and fused SwiGLU pairs (Neutrino-1 8B
// model page: seven coded linears per layer, gate/up feeding a SwiGLU; the
// speculative verifier's M = 7 pass), optionally behind an RMSNorm of their
// activations (spec table); and, as a second instantiation of the same
// kernel, the int8 output head with the greedy argmax fused ("Where the
// bytes live"; the spec-decode paragraph's greedy acceptance).
//
// Each of the grid's CTAs (one per SM) owns a contiguous run of work units;
// a unit is one 128-row tile (64 gate + 64 up rows for a SwiGLU pair) of one
// item over the item's whole K, so no unit needs a cross-CTA reduction.  The
// host balances the runs by packed bytes.  K is processed in chunks whose
// one-band B fits a 56 KB buffer (the whole K for m = 1 at every Neutrino
// shape).  The B operand holds each activation as two e4m3 terms (hi, lo)
// under a per-row power-of-two scale per chunk; a chunk where small
// elements would matter (outlier channels) takes two magnitude bands, four
// terms, across both buffers (split_word2).  B and the fp32 accumulators
// are double buffered per chunk; a one-band chunk's B is reused by every
// later tile of the item on the same buffer, and fetching the next chunk's
// B and reading the previous chunk's sums overlap the weight stream.
// Roles (17 warps):
//   * warp 0, lane 0: TMA producer; streams every stage of every unit of the
//     CTA through a 6-deep ring of 16 KB stages (128 rows x 512 codes, or
//     x 128 int8 weights; 128-byte swizzle), never waiting on activations.
//   * warps 1-4: bring in B for each chunk (after griddepcontrol.wait), then
//     read the previous chunk's accumulators, rescale and add them into
//     per-row registers, and at the end of a unit write y (scale, SiLU gate;
//     int8 head: logits and the argmax keys).  For m = 1 they build B from x
//     themselves (normalising it first for items with a norm); for m >= 2 a
//     short kernel launched just before (k_tern_bprep) has written every
//     chunk's one-band B, row maxima and band flags to a workspace once, and
//     a one-band chunk is one bulk copy: building it in every CTA that
//     streams a tile of the item costs more than the chunk's weight stream
//     when m is large.
//   * warps 5-16: three decoder groups of four warps; group g turns the four
//     chunk columns (128 codes of a row each) of the stages s = g (mod 3)
//     into e4m3 +-2/0 bytes (decode8) in TMEM slot g, and lane 0 of warp q
//     of the group then issues the K = 32 steps of column q (tcgen05.mma
//     kind::f8f6f4, A from TMEM, B from shared memory, M = 128) into the
//     column's accumulator of the chunk's buffer.  One-band chunks take the
//     fixed N = 16 path; two-band chunks an out-of-line one (N = 16 for
//     m <= 4; N = 32 for m >= 5 as two 256-code columns from quads 0 and
//     1).  Three decoder warps per scheduler hide each other's barrier
//     latency.  The int8 format decodes each weight into two exact e4m3
//     nibbles and issues one MMA per nibble and K step (see kFmtI8).
// Every mbarrier wait is bounded; on time-out the kernel records the error,
// stops, drains its copies and MMAs, releases its tensor memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <utility>
#include <vector>

#include "tern.h"
#include "tern_internal.cuh"
#include "tern_mma_common.cuh"
#include "tern_ptx.cuh"

namespace tern {

namespace {

using namespace mma;

constexpr int kMaxItems = 128;             // items per launch (kernel parameter space)
constexpr int kMaxMaps = 144;              // tensor maps per launch: one per item, two per SwiGLU pair
constexpr int kMaxCtas = 160;
constexpr int kThreads = 544;              // 17 warps
constexpr int kFirstStager = 1;            // warps 1-4
constexpr int kStagers = 128;
constexpr int kFirstDec = 5;               // warps 5-16: three decoder groups of four warps
constexpr int kCols = 4;                   // chunk columns of a stage; warp q of a group issues column q
// Decoder group g decodes the stages s = g (mod 3) into TMEM slot g and ring
// slots g and g + 3: every slot a group waits on was last used by the group
// itself, so a phase-parity wait can never be two phases ahead (which would
// alias).
constexpr int kDecGroups = 3;
constexpr int kASlots = 3;                 // TMEM A slots, one stage (128 columns) each
constexpr uint32_t kTmemCols = 512;
// Accumulators: 128 columns from kDCol, two buffers of 64 that alternate
// chunk by chunk.  N = 16 (m <= 4): D[buf][q] at kDCol + 16 * (4 buf + q) for
// the four 128-code columns q of a stage.  N = 32 (m >= 5): D[buf][q] at
// kDCol + 32 * (2 buf + q) for two 256-code columns.
constexpr uint32_t kDCol = kASlots * 128;
// Weight formats of the persistent kernel: the ternary 2-bit codes (a stage
// is 512 codes of a row, 32 activation words of 16), and the int8 output
// head (a stage is 128 weights of a row, 8 activation words).  For int8 each
// weight b = 16 (h - 8) + l with h, l in [0, 15] (offset binary), and both
// nibbles enter the MMA as e4m3 bytes whose value is nibble * 2^-9 (the
// e4m3 bytes 0x00..0x0F are exactly v * 2^-9): TMEM slot g holds the l
// bytes of a stage in columns 64g .. 64g + 31 and the h bytes in 64g + 32 ..
// 64g + 63, and each of the four chunk columns (one K = 32 step each) has
// an accumulator per nibble, D_l[buf][q] at kDColL + 16 (4 buf + q) and
// D_h at kDColH + 16 (4 buf + q).
constexpr int kFmtTern = 0;
constexpr int kFmtI8 = 1;
constexpr uint32_t kDColL = 256;
constexpr uint32_t kDColH = 384;
__host__ __device__ constexpr int stage_b_words(int fmt) { return fmt == kFmtI8 ? 8 : kStageWords; }
// Two B buffers, contiguous, then the MMA's read slack.  A chunk is planned
// so that its one-band operand (b_block_bytes(m, 1) per 16-code block) fits
// one buffer; a chunk that needs two bands (twice the bytes) takes both
// buffers, starting at the first.
#ifndef TERN_BBUF_KB
#define TERN_BBUF_KB 56
#endif
constexpr int kBBufBytes = TERN_BBUF_KB * 1024;
// Weight ring depth: 96 KB in flight per SM covers DRAM latency at the HBM
// rate (a plain TMA stream of these stages runs as fast with 6 as with 9);
// the rest of shared memory goes to the two 56 KB activation buffers.  The
// depth is a multiple of kDecGroups (see there).
#ifndef TERN_WSTAGES
#define TERN_WSTAGES 6
#endif
constexpr int kWStages = TERN_WSTAGES;

struct Item {
    const float *scale_g;
    const float *scale_u;
    const uint16_t *x;
    float *y;
    int rows, k, m, swiglu;
    int stages;  // 512-code stages over K
    int cstages; // stages per K chunk (the last may be shorter); a chunk's B fits one buffer
    int unit0;   // first global unit of this item
    int map;     // its codes' tensor map (gate, then up, for a SwiGLU pair)
    // B prepared by k_tern_bprep (m >= 2; nullptr for m = 1): the one-band
    // compact layout of the padded K (word w of row i at w * 32m + 32i), so
    // chunk c starts at byte c * cstages * 1024m; meta[kMetaWords * c ...]
    // holds its rows' maxima and band-B flags.
    const unsigned char *bsrc;
    const uint32_t *meta;
    const float *norm_w;  // RMSNorm channel weights [k], or nullptr: x enters as given
};

struct Params {
    int n_items;
    float eps;                     // RMSNorm eps of the items with norm weights
    long long wait_limit;          // bound of every Waiter, in cycles
    unsigned long long *keys;      // int8 head: per activation row the best (logit, index) key so far
    int unit_start[kMaxCtas + 1];  // CTA b runs units [unit_start[b], unit_start[b + 1])
    int item_start[kMaxCtas];      // the item holding unit unit_start[b]
    int stages_cta[kMaxCtas];      // 512-code stages in CTA b's run
    Item item[kMaxItems];
};

struct Maps {
    CUtensorMap m[kMaxMaps];
};

// Shared-memory layout (bytes from the 1024-aligned base).
constexpr uint32_t kOffW = 0;
constexpr uint32_t kOffB = kOffW + kWStages * kStageBytes;
constexpr uint32_t kOffXch = kOffB + 2 * kBBufBytes + kBPad;  // [64][8] fp32
constexpr uint32_t kOffBar = kOffXch + 64 * 8 * 4;
constexpr uint32_t kBarWFull = 0;                       // [kWStages]
constexpr uint32_t kBarWEmpty = kBarWFull + 8 * kWStages;
constexpr uint32_t kBarAEmpty = kBarWEmpty + 8 * kWStages;  // [kASlots]: the slot's MMAs are done
constexpr uint32_t kBarBFull = kBarAEmpty + 8 * kASlots;     // [2]
constexpr uint32_t kBarBEmpty = kBarBFull + 16;
constexpr uint32_t kBarDFull = kBarBEmpty + 16;
constexpr uint32_t kBarDEmpty = kBarDFull + 16;
constexpr uint32_t kBarDrain = kBarDEmpty + 16;  // one commit per issuing warp on exit
constexpr uint32_t kBarTurn = kBarDrain + 8;     // [kCols][kDecGroups]: group g's turn on column q
constexpr uint32_t kWordsOff = kBarTurn + 8 * kCols * kDecGroups;
// words: [0] tmem base, [1] abort, [8..39] B buffer 0's chunk metadata,
// [40..71] buffer 1's: per activation row i, [2i] row maximum and [2i + 1]
// band-B maximum; [16] the chunk's number times 4 plus its band count; [17],
// [18] scratch of the m = 1 build; [24 + i] row i's RMSNorm factor (fp32
// bits; items with a norm); [32 + 2i], [33 + 2i] the chunk's sum of row i's
// activations as an fp32 pair (int8 head)
constexpr uint32_t kWordsCount = 104;
constexpr uint32_t kXmWords = 48;
constexpr uint32_t kSmemBytes = 1024 + kOffBar + kWordsOff + kWordsCount * 4;

__device__ unsigned int g_batched_error;

// Walks the (unit, chunk) sequence of one CTA.  A CTA's units are
// contiguous, so the item index only moves forward; the fields of the current
// item live in registers (a dependent search through the parameter space on
// every unit costs more than a stage of decoding).
struct Cursor {
    const Params *p;
    int unit, unit_end, item, next_unit0, tile, chunk, n_chunks, stages, cstages, n_stages_chunk;
    __device__ void enter_item()
    {
        stages = p->item[item].stages;
        cstages = p->item[item].cstages;
        n_chunks = (stages + cstages - 1) / cstages;
        next_unit0 = item + 1 < p->n_items ? p->item[item + 1].unit0 : 0x7FFFFFFF;
    }
    __device__ void set_chunk() { n_stages_chunk = min(cstages, stages - chunk * cstages); }
    __device__ bool begin(const Params *pp, int b)
    {
        p = pp;
        unit = p->unit_start[b];
        unit_end = p->unit_start[b + 1];
        if (unit >= unit_end) return false;
        item = p->item_start[b];
        enter_item();
        tile = unit - p->item[item].unit0;
        chunk = 0;
        set_chunk();
        return true;
    }
    // Advance one chunk; false at the end of the CTA's run.
    __device__ bool next_chunk()
    {
        if (++chunk < n_chunks) {
            set_chunk();
            return true;
        }
        if (++unit >= unit_end) return false;
        chunk = 0;
        ++tile;
        if (unit >= next_unit0) {  // every item has at least one unit
            ++item;
            enter_item();
            tile = 0;
        }
        set_chunk();
        return true;
    }
    __device__ bool last_chunk_of_unit() const { return chunk + 1 == n_chunks; }
};

// ------------------------------------------------------------------ B prep
// One CTA per (item, chunk, activation row) of the items with m >= 2: the
// row's largest |x| over the chunk; below the band threshold it sets, the
// largest |x| (band B), the count of nonzero elements and the sum of all
// |x|, and from these whether the row needs band B (need_two_bands); then
// every word (16 k) of the row split into its one-band e4m3 rows
// (split_word1), written in the compact layout the MMA reads (Item::bsrc,
// words past K zero).  A chunk holds at most 28 stages (m = 2), so each
// thread keeps its words in registers and all loads are in flight at once.
// A chunk in which some row needs band B is built by the persistent kernel
// from x and these maxima instead (rare: activations with outlier channels).
constexpr int kPrepThreads = 128;
constexpr int kPrepWords = 7;           // words per thread: 28 stages * 32 / 128
constexpr uint32_t kBulkPiece = 16384;  // bytes per bulk copy of a prepared chunk
// Per-chunk metadata (48 words): for activation row i, [2i] its maximum and
// [2i + 1] its band-B maximum (fp32 bits of |x|), [16 + i] 1 if it needs
// band B, [24 + i] its RMSNorm factor (items with a norm), [32 + 2i] and
// [33 + 2i] the sum of its activations over the chunk as an fp32 pair (int8
// head).
constexpr int kMetaWords = 48;

struct PrepItem {
    const uint16_t *x;
    const float *norm_w;  // RMSNorm channel weights [k], or nullptr
    int sw;               // activation words per stage (stage_b_words)
    int head;             // int8 head: B in k order, and the chunk's activation sums
    unsigned char *b;
    uint32_t *meta;
    int k, m, stages, cstages;
    int task0;  // first task of the item; task task0 + c * m + i is chunk c, row i
};

struct PrepParams {
    int n_items, n_tasks;
    float eps;
    PrepItem item[kMaxItems];
};

// Maximum of v over the CTA of k_tern_bprep; every thread gets it.
__device__ __forceinline__ uint32_t prep_cta_max(uint32_t v, uint32_t *red)
{
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kPrepThreads / 32; ++w) v = max(v, red[w]);
    __syncthreads();  // red is reused by the next reduction
    return v;
}

__global__ void __launch_bounds__(kPrepThreads) k_tern_bprep(const __grid_constant__ PrepParams p)
{
    __shared__ uint32_t red[kPrepThreads / 32];
    __shared__ uint32_t stat[kPrepThreads / 32][3];
    __shared__ double ssred[kPrepThreads / 32];
    // The persistent kernel that follows may start at once: its weight stream
    // needs nothing from here, and its staging warps wait for this grid to
    // finish before they read the workspace.  The previous kernel on the
    // stream may still read the workspace, and x may come from it: wait for
    // it.
    ptx::grid_dep_launch();
    ptx::grid_dep_wait();
    const int tid = (int)threadIdx.x, task = (int)blockIdx.x;
    int j = 0;
    while (j + 1 < p.n_items && p.item[j + 1].task0 <= task) ++j;
    const PrepItem &it = p.item[j];
    const int local = task - it.task0, c = local / it.m, mm = local - c * it.m;
    const int w0 = c * it.cstages * it.sw;
    const int nw = min(it.cstages, it.stages - c * it.cstages) * it.sw;
    const int kw = it.k / 16;
    // Word slots a thread uses: every loop over the slots stops at nq (the
    // same for the whole CTA), so a chunk shorter than the largest one runs
    // only the code of its own slots.  Each CTA passes through the code once,
    // so the instructions it executes are mostly fetched cold.
    const int nq = (nw + kPrepThreads - 1) / kPrepThreads;
    const uint4 *xr = reinterpret_cast<const uint4 *>(it.x + (size_t)mm * it.k);  // 2 x uint4 per word
    uint4 va[kPrepWords], vb[kPrepWords];
#pragma unroll
    for (int q = 0; q < kPrepWords; ++q) {
        const int wi = tid + q * kPrepThreads, gw = w0 + wi;
        va[q] = vb[q] = make_uint4(0u, 0u, 0u, 0u);
        if (q < nq && wi < nw && gw < kw) {
            va[q] = __ldg(xr + 2 * gw);
            vb[q] = __ldg(xr + 2 * gw + 1);
        }
    }
    float rn = 0.f;
    if (it.norm_w != nullptr) {
        // RMSNorm: the mean square over the whole row (every chunk's CTA of
        // the row takes it), then this chunk's words normalised in place
        double ss = 0.0;
        for (int w = tid; w < kw; w += kPrepThreads) ss += sumsq16(__ldg(xr + 2 * w), __ldg(xr + 2 * w + 1));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
        if ((tid & 31) == 0) ssred[tid >> 5] = ss;
        __syncthreads();
        ss = 0.0;
#pragma unroll
        for (int w = 0; w < kPrepThreads / 32; ++w) ss += ssred[w];
        rn = rms_factor(ss, it.k, p.eps);
        const float4 *g4 = reinterpret_cast<const float4 *>(it.norm_w);
#pragma unroll
        for (int q = 0; q < kPrepWords; ++q) {
            if (q >= nq) break;
            const int wi = tid + q * kPrepThreads, gw = w0 + wi;
            if (wi < nw && gw < kw) rmsnorm_word(va[q], vb[q], g4 + 4 * gw, rn);
        }
    }
    uint32_t mx = 0;
#pragma unroll
    for (int q = 0; q < kPrepWords; ++q) {
        if (q >= nq) break;
        mx = max(mx, max_abs16(va[q], vb[q]));
    }
    const uint32_t ma = prep_cta_max(mx, red);
    const uint32_t tb2 = band_threshold2(ma);
    uint32_t n = 0, mb = 0;
    float sabs = 0.f;
#pragma unroll
    for (int q = 0; q < kPrepWords; ++q) {
        if (q >= nq) break;
        band_stats16(va[q], vb[q], tb2, n, sabs);
        mb = max(mb, max_abs16_below(va[q], vb[q], tb2));
    }
    // the three statistics over the CTA in one round
    mb = __reduce_max_sync(0xFFFFFFFFu, mb);
    n = __reduce_add_sync(0xFFFFFFFFu, n);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sabs += __shfl_xor_sync(0xFFFFFFFFu, sabs, o);
    if ((tid & 31) == 0) {
        stat[tid >> 5][0] = mb;
        stat[tid >> 5][1] = n;
        stat[tid >> 5][2] = __float_as_uint(sabs);
    }
    __syncthreads();
    mb = n = 0;
    sabs = 0.f;
#pragma unroll
    for (int w = 0; w < kPrepThreads / 32; ++w) {
        mb = max(mb, stat[w][0]);
        n += stat[w][1];
        sabs += __uint_as_float(stat[w][2]);
    }
    if (it.head) {
        double sx = 0.0;
#pragma unroll
        for (int q = 0; q < kPrepWords; ++q) {
            if (q >= nq) break;
            sx += sum16(va[q], vb[q]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sx += __shfl_xor_sync(0xFFFFFFFFu, sx, o);
        __syncthreads();  // ssred free
        if ((tid & 31) == 0) ssred[tid >> 5] = sx;
        __syncthreads();
        if (tid == 0) {
            sx = 0.0;
            for (int w = 0; w < kPrepThreads / 32; ++w) sx += ssred[w];
            const float hi = (float)sx;
            uint32_t *meta = it.meta + (size_t)kMetaWords * c;
            meta[32 + 2 * mm] = __float_as_uint(hi);
            meta[33 + 2 * mm] = __float_as_uint((float)(sx - (double)hi));
        }
    }
    if (tid == 0) {
        uint32_t *meta = it.meta + (size_t)kMetaWords * c;
        meta[2 * mm] = ma;
        meta[2 * mm + 1] = mb;
        meta[16 + mm] = need_two_bands(ma, n, sabs) ? 1u : 0u;
        meta[24 + mm] = __float_as_uint(rn);
    }
    const float sc = exp2i(row_scale_exp(ma));
    const size_t wbytes = b_block_bytes(it.m, 1);
    unsigned char *dst = it.b + (size_t)w0 * wbytes + 32u * (size_t)mm;
#pragma unroll
    for (int q = 0; q < kPrepWords; ++q) {
        if (q >= nq) break;
        const int wi = tid + q * kPrepThreads;
        if (wi < nw) {
            uint4 rows[2];
            split_word1(va[q], vb[q], sc, rows, it.head != 0);
            uint4 *d = reinterpret_cast<uint4 *>(dst + (size_t)wi * wbytes);
            d[0] = rows[0];
            d[1] = rows[1];
        }
    }
}

// The MMAs of one stage's column `quad` for a chunk with two bands (4m B
// rows per 16-code block, both B buffers from the first): N = 16 for m <= 4,
// with four 128-code columns; N = 32 for m >= 5, with two 256-code columns
// issued by quads 0 and 1 (quads 2 and 3 issue nothing).  Kept out of line:
// it runs only for activations with outlier channels.
__device__ __noinline__ void issue_two_band(uint32_t tmem, uint32_t bbuf, int g, int quad, int buf, int st, int m)
{
    const int n = mma_n(m, 2);
    const int cols = n == 32 ? 2 : kCols;
    if (quad >= cols) return;
    const int steps = 16 / cols;  // K = 32 steps per column
    const uint32_t wbytes = b_block_bytes(m, 2);
    const uint32_t idesc = idesc_n(n);
    const uint32_t d = tmem + kDCol + (uint32_t)(n * (cols * buf + quad));
    const uint32_t a = tmem + (uint32_t)(g * 128 + quad * 8 * steps);
    const uint64_t bd = b_desc_lbo(bbuf + (uint32_t)(st * kStageWords + 2 * steps * quad) * wbytes, wbytes);
    const uint32_t bd_lo = (uint32_t)bd, bd_hi = (uint32_t)(bd >> 32), t_step = (2u * wbytes) >> 4;
    for (int t = 0; t < steps; ++t)
        ptx::mma_ts_f8f6f4_lh(d, a + 8u * (uint32_t)t, bd_lo + t_step * (uint32_t)t, bd_hi, idesc,
                              (st != 0 || t != 0) ? 1u : 0u);
}

// int8 head: the MMAs of one stage's column `quad` for a chunk with two
// bands (N = 16 for m <= 4 with four one-step columns; N = 32 for m >= 5 with
// two two-step columns issued by quads 0 and 1), both nibbles of each step.
__device__ __noinline__ void issue_two_band_i8(uint32_t tmem, uint32_t bbuf, int g, int quad, int buf, int st, int m)
{
    const int n = mma_n(m, 2);
    const int cols = n == 32 ? 2 : kCols;
    if (quad >= cols) return;
    const int steps = 4 / cols;  // K = 32 steps per column
    const uint32_t wbytes = b_block_bytes(m, 2);
    const uint32_t idesc = idesc_n(n);
    const uint32_t dl = tmem + kDColL + (uint32_t)(n * (cols * buf + quad)), dh = dl + (kDColH - kDColL);
    for (int t = 0; t < steps; ++t) {
        const int ks = quad * steps + t;
        const uint32_t al = tmem + (uint32_t)(g * 64 + 8 * ks);
        const uint64_t bd = b_desc_lbo(bbuf + (uint32_t)(st * stage_b_words(kFmtI8) + 2 * ks) * wbytes, wbytes);
        const uint32_t acc = (st != 0 || t != 0) ? 1u : 0u;
        ptx::mma_ts_f8f6f4_lh(dl, al, (uint32_t)bd, (uint32_t)(bd >> 32), idesc, acc);
        ptx::mma_ts_f8f6f4_lh(dh, al + 32u, (uint32_t)bd, (uint32_t)(bd >> 32), idesc, acc);
    }
}

// One stage of one int8 row (128 weights in 8 words, after the swizzle) ->
// its TMEM A rows: the low nibbles l = b & 15 in the first 32 columns, the
// offset high nibbles h = ((b ^ 0x80) >> 4) in the next 32, each as the e4m3
// byte of value nibble * 2^-9.
__device__ __forceinline__ void decode_i8_stage(uint32_t srow, uint32_t sw, uint32_t ta)
{
#pragma unroll
    for (int half = 0; half < 2; ++half) {  // 64 weights: TMEM columns 16 half .. 16 half + 15 of each nibble
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 v = ptx::lds128(srow + ((((uint32_t)(4 * half + c)) ^ sw) << 4));
            w[4 * c] = v.x;
            w[4 * c + 1] = v.y;
            w[4 * c + 2] = v.z;
            w[4 * c + 3] = v.w;
        }
        uint32_t r[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) r[j] = w[j] & 0x0F0F0F0Fu;
        ptx::tmem_st_32x32b_x16(ta + 16u * (uint32_t)half, r);
#pragma unroll
        for (int j = 0; j < 16; ++j) r[j] = ((w[j] >> 4) ^ 0x08080808u) & 0x0F0F0F0Fu;
        ptx::tmem_st_32x32b_x16(ta + 32u + 16u * (uint32_t)half, r);
    }
}

template <int kFmt>
__global__ void __launch_bounds__(kThreads, 1)
k_tern_batched(const __grid_constant__ Params p, const __grid_constant__ Maps maps)
{
    constexpr bool kI8 = kFmt == kFmtI8;
    constexpr int kSW = stage_b_words(kFmt);  // activation words per stage
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *gbase = smem_raw + (base - raw);
    const uint32_t wbuf = base + kOffW;
    const uint32_t bbuf = base + kOffB;
    float *xch = reinterpret_cast<float *>(gbase + kOffXch);
    const uint32_t bars = base + kOffBar;
#ifdef TERN_WAIT_DIAG
    if (threadIdx.x == 0 && blockIdx.x == 0) printf("k_tern_batched barriers at %u\n", bars);
#endif
    uint32_t *words = reinterpret_cast<uint32_t *>(gbase + kOffBar + kWordsOff);
    volatile uint32_t *abort_flag = words + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < kWStages; ++s) {
            ptx::mbar_init(bars + kBarWFull + 8 * s, 1);
            ptx::mbar_init(bars + kBarWEmpty + 8 * s, 4 * 32);  // every lane of the stage's decoder group
        }
        for (int s = 0; s < kASlots; ++s) ptx::mbar_init(bars + kBarAEmpty + 8 * s, kCols);  // the group's issuing lanes
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bars + kBarBFull + 8 * b, kStagers);  // every staging thread, after its proxy fence
            ptx::mbar_init(bars + kBarBEmpty + 8 * b, kCols);  // the issuing lanes of the chunk's last stage
            ptx::mbar_init(bars + kBarDFull + 8 * b, kCols);
            ptx::mbar_init(bars + kBarDEmpty + 8 * b, 4);
        }
        ptx::mbar_init(bars + kBarDrain, kDecGroups * kCols);
        for (int j = 0; j < kCols * kDecGroups; ++j) ptx::mbar_init(bars + kBarTurn + 8 * j, 1);
        for (int j = 1; j < (int)kWordsCount; ++j) words[j] = 0u;
        // no chunk's tag in the band words yet (a zero word would read as chunk 0's)
        words[8 + 16] = words[8 + kXmWords + 16] = ~0u;
        ptx::fence_proxy_async_smem();
    }
    if (warp == 0) {
        __syncwarp();
        ptx::tmem_alloc(ptx::smem_u32(words), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = words[0];
    if (tid == 0) ptx::grid_dep_launch();
    const Waiter waiter(abort_flag, &g_batched_error, p.wait_limit);
    Cursor cur;
    const bool any = cur.begin(&p, (int)blockIdx.x);

    if (warp == 0) {
        // --------------------------------------------------------- producer
        // "Empty" barriers are waited at the flipped parity: a fresh barrier
        // counts its preceding phase as complete, so the first pass through
        // the ring needs no special case.
        if (lane == 0 && any) {
            int gs = 0, slot = 0;
            uint32_t par = 0;
            bool more = true;
            while (more) {
                const Item &it = p.item[cur.item];
                const int row0 = cur.tile * (it.swiglu ? 64 : 128);
                for (int st = 0; st < cur.n_stages_chunk; ++st, ++gs) {
                    const uint32_t empty = bars + kBarWEmpty + 8 * slot;
                    if (!ptx::mbar_try_wait(empty, par ^ 1u) && !waiter.wait(empty, par ^ 1u)) {
                        more = false;
                        break;
                    }
                    const uint32_t dst = wbuf + slot * kStageBytes, full = bars + kBarWFull + 8 * slot;
                    const int c0 = (cur.chunk * cur.cstages + st) * kStageWords;
                    ptx::mbar_arrive_expect_tx(full, kStageBytes);
                    ptx::tma_load_2d(dst, &maps.m[it.map], c0, row0, full);
                    if (it.swiglu) ptx::tma_load_2d(dst + kStageBytes / 2, &maps.m[it.map + 1], c0, row0, full);
                    if (++slot == kWStages) {
                        slot = 0;
                        par ^= 1u;
                    }
                }
                more = more && cur.next_chunk();
            }
            for (int s = gs > kWStages ? gs - kWStages : 0; s < gs; ++s)
                drain_wait(bars + kBarWFull + 8 * (s % kWStages), (s / kWStages) & 1, &g_batched_error);
        }
    } else if (warp >= kFirstDec) {
        // ----------------------------------------- decoders and MMA issuers
        // Group g decodes all four columns of the stages s = g (mod 3) into
        // TMEM slot g (quad q owns TMEM lanes 32q..32q+31), the group meets
        // at a named barrier, and then warp q issues the four K=32 steps of
        // column q (tcgen05.mma kind::f8f6f4, A from TMEM, B from shared
        // memory, M = 128, N = 16 or 32) into D[buf][q].  Stage s's MMAs on a column
        // follow stage s-1's, issued by the previous group, through that
        // column's turn barriers (tcgen05 fence, mbarrier, fence), which order
        // the accumulation; a warp issues for one stage in three, so one
        // thread's waits and bookkeeping overlap the others' MMA issue (a
        // warp issues an MMA about every 54 cycles, warps overlap).  Every
        // slot a group waits on was last used by the group itself, so no
        // phase-parity wait runs two phases ahead of its barrier.  A chunk's
        // first-stage issuers wait for its B buffer and for the epilogue
        // that last read its accumulator columns (later stages see both
        // through the turn chain); its last-stage issuers commit the chunk's
        // D and B, which tracks the whole accumulation chain.
        const int g = (warp - kFirstDec) >> 2;
        const int quad = warp & 3;
        const int i = quad * 32 + lane;
        const uint32_t tm_row = tmem + ((uint32_t)(quad * 32) << 16);
        const uint32_t row_addr = wbuf + (uint32_t)i * 128u;
        const uint32_t sw = (uint32_t)(i & 7);  // 128-byte swizzle: 16-byte chunk c of row i sits at c ^ (i & 7)
        const uint32_t my_turn = bars + kBarTurn + 8u * (uint32_t)(kDecGroups * quad + g);
        const uint32_t next_turn = bars + kBarTurn + 8u * (uint32_t)(kDecGroups * quad + (g + 1) % kDecGroups);
        const uint32_t a_empty = bars + kBarAEmpty + 8u * (uint32_t)g;
        const uint32_t bar_id = 2u + (uint32_t)g;  // 0: __syncthreads, 1: staging warps
        static_assert(kWStages % kDecGroups == 0 && kASlots == kDecGroups, "slots must cycle within a group");
        int w_r = g, w_q = 0;      // stage s: ring slot s % kWStages, use s / kWStages
        int a_q = 0;               //          TMEM slot g, use s / kASlots
        uint32_t tpar = g == 0 ? 1u : 0u;  // stage 0 needs no turn
        int gs = 0, gc = 0;
        uint32_t bw = 0;  // band word of chunk bw_gc
        int bw_gc = -1;
        bool more = any;
        while (more) {
            const int n_st = cur.n_stages_chunk;
            const int buf = gc & 1;
            const int m = p.item[cur.item].m;
            // The epilogue that last read this buffer's accumulators (chunk
            // gc - 2's) must be done; for gc < 2 that is the phase a fresh
            // barrier counts as complete.
            const uint32_t dempty = bars + kBarDEmpty + 8u * (uint32_t)buf;
            const uint32_t dpar = ((uint32_t)(gc >> 1) & 1u) ^ 1u;
            for (int st = (g - gs % kDecGroups + kDecGroups) % kDecGroups; st < n_st; st += kDecGroups) {
                const uint32_t wf = bars + kBarWFull + 8 * w_r;
                const uint32_t wpar = (uint32_t)w_q & 1u, apar = (uint32_t)a_q & 1u;
                // both fast-path tests issue back to back; the bounded waits only on a miss
                bool okw = ptx::mbar_try_wait(wf, wpar);
                bool oka = ptx::mbar_try_wait(a_empty, apar ^ 1u);
                if (!okw) okw = waiter.wait(wf, wpar);
                if (okw && !oka) oka = waiter.wait(a_empty, apar ^ 1u);
                if (__all_sync(0xFFFFFFFFu, okw && oka)) {
                    ptx::tc_fence_after();
                    const uint32_t srow = row_addr + (uint32_t)w_r * kStageBytes;
                    if constexpr (kI8) {
                        decode_i8_stage(srow, sw, tm_row + (uint32_t)(g * 64));
                    } else {
                        const uint32_t ta = tm_row + (uint32_t)(g * 128);
#pragma unroll 1
                        for (int c = 0; c < 4; ++c) {
                            const uint4 v0 = ptx::lds128(srow + ((((uint32_t)(2 * c)) ^ sw) << 4));
                            const uint4 v1 = ptx::lds128(srow + ((((uint32_t)(2 * c + 1)) ^ sw) << 4));
                            uint32_t r[32];
                            decode8(v0, v1, r);
                            ptx::tmem_st_32x32b_x32(ta + 32u * (uint32_t)c, r);
                        }
                    }
                    ptx::mbar_arrive(bars + kBarWEmpty + 8 * w_r);  // after the last store, which consumed the loads
                    ptx::tmem_wait_st();
                }
                ptx::tc_fence_before();
                // the group's 128 rows are in TMEM; stop together on an abort
                if (ptx::named_bar_or(bar_id, 128, *abort_flag != 0u)) {
                    more = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t bpar = (uint32_t)(gc >> 1) & 1u;
                    const uint32_t bfull = bars + kBarBFull + 8 * buf;
                    // The turn first: once it has come, chunk gc - 2 (the same B
                    // buffer) has passed its own BFull wait and the epilogue
                    // before the one waited for here is done, so neither
                    // parity wait below can run ahead of its barrier (a wait
                    // one phase early returns at once, taking the earlier
                    // phase for this one).
                    bool lok = ptx::mbar_try_wait(my_turn, tpar) || waiter.wait(my_turn, tpar);
                    lok = lok && (st != 0 || ((ptx::mbar_try_wait(bfull, bpar) || waiter.wait(bfull, bpar)) &&
                                              (ptx::mbar_try_wait(dempty, dpar) || waiter.wait(dempty, dpar))));
                    if (lok) {
                        ptx::tc_fence_after();
                        // The chunk's band count, written by the staging warps
                        // before their BFull arrival, read once per chunk: the
                        // stage-0 issuer waited for BFull and every later
                        // stage's issuer follows it through the turn chain,
                        // while the word is rewritten only after this chunk's
                        // last stage has been issued.
                        if (bw_gc != gc) {
                            bw = words[8 + kXmWords * buf + 16];
                            bw_gc = gc;
                        }
                        if constexpr (kI8) {
                            if ((bw & 3u) != 2u) {
                                // one band, N = 16: column q is K step q of the
                                // stage, one MMA per nibble
                                const uint32_t wbytes = b_block_bytes(m, 1);
                                const uint32_t dl = tmem + kDColL + 16u * (uint32_t)(kCols * buf + quad);
                                const uint32_t al = tmem + (uint32_t)(g * 64 + 8 * quad);
                                const uint64_t bd = b_desc_lbo(bbuf + (uint32_t)buf * kBBufBytes +
                                                                   (uint32_t)(st * kSW + 2 * quad) * wbytes,
                                                               wbytes);
                                constexpr uint32_t kIdesc16 = idesc_n(16);
                                const uint32_t acc = st != 0 ? 1u : 0u;
                                ptx::mma_ts_f8f6f4_lh(dl, al, (uint32_t)bd, (uint32_t)(bd >> 32), kIdesc16, acc);
                                ptx::mma_ts_f8f6f4_lh(dl + (kDColH - kDColL), al + 32u, (uint32_t)bd,
                                                      (uint32_t)(bd >> 32), kIdesc16, acc);
                            } else {
                                issue_two_band_i8(tmem, bbuf, g, quad, buf, st, m);
                            }
                        } else if ((bw & 3u) != 2u) {
                            // one band: N = 16 (2m <= 16); compact B, column q
                            // of stage st at word st*32 + 8q, its K = 32 step t
                            // at A column +8t and B word +2t
                            const uint32_t wbytes = b_block_bytes(m, 1);
                            const uint32_t d = tmem + kDCol + 16u * (uint32_t)(kCols * buf + quad);
                            const uint32_t a = tmem + (uint32_t)(g * 128 + quad * 32);
                            const uint64_t bd = b_desc_lbo(bbuf + (uint32_t)buf * kBBufBytes +
                                                               (uint32_t)(st * kStageWords + 8 * quad) * wbytes,
                                                           wbytes);
                            const uint32_t bd_lo = (uint32_t)bd, bd_hi = (uint32_t)(bd >> 32);
                            const uint32_t t_step = (2u * wbytes) >> 4;
                            constexpr uint32_t kIdesc16 = idesc_n(16);
                            ptx::mma_ts_f8f6f4_lh(d, a, bd_lo, bd_hi, kIdesc16, st != 0 ? 1u : 0u);
#pragma unroll
                            for (int t = 1; t < 4; ++t)
                                ptx::mma_ts_f8f6f4_lh(d, a + 8u * t, bd_lo + t_step * t, bd_hi, kIdesc16, 1u);
                        } else {
                            issue_two_band(tmem, bbuf, g, quad, buf, st, m);
                        }
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(next_turn);  // the next stage's MMAs on this column follow these
                        ptx::mma_commit(a_empty);
                        if (st == n_st - 1) {
                            ptx::mma_commit(bars + kBarDFull + 8 * buf);
                            ptx::mma_commit(bars + kBarBEmpty + 8 * buf);
                        }
                    }
                }
                __syncwarp();
                tpar ^= 1u;
                w_r += kDecGroups;  // s += 3
                if (w_r >= kWStages) {
                    w_r -= kWStages;
                    ++w_q;
                }
                ++a_q;
            }
            gs += n_st;
            ++gc;
            more = more && cur.next_chunk();
        }
        // arrives once every MMA this thread issued has completed (at once if none)
        if (lane == 0) ptx::mma_commit(bars + kBarDrain);
    } else {
        // ------------------------------------------- B staging and epilogue
        const int st_tid = tid - 32 * kFirstStager;  // 0..127
        const int quad = warp & 3;
        const int i = quad * 32 + lane;               // tile row == TMEM lane
        ptx::grid_dep_wait();
        // Per activation row, the unit's sum so far.  While every chunk of the
        // unit has had one band it is a plain fp32 sum: the band choice
        // already keeps each chunk within 2^-24 of its sum|x|.  From the first
        // two-band chunk on (outlier channels, whose partial sums may cancel
        // far below their own size) it is an unevaluated pair (acc_pair).
        float acc[8], acc_lo[8];
        bool pairs = false;
#pragma unroll
        for (int n = 0; n < 8; ++n) acc[n] = acc_lo[n] = 0.f;
        // previous chunk, whose accumulators are read after the next chunk's B is staged
        int prev_item = -1, prev_tile = 0, prev_bands = 1;
        bool prev_last = false;
        int gc = 0;
        bool ok = any;
        // what each B buffer holds: a one-band chunk of an item is staged once
        // and reused by every later tile of the same item that lands on it
        int held_item[2] = {-1, -1}, held_chunk[2] = {-1, -1};
        int last_gc[2] = {-1, -1};  // last chunk whose BFull phase each buffer took part in
        uint32_t *meta_s = words + 8;  // [kXmWords] per buffer: row maxima, then the band count at [16]

        // Reads chunk e's accumulators into the rows' pairs and finishes the
        // unit if it was its last chunk.  Within a band the issuing columns
        // and the hi/lo terms are summed in fp32 (one band, one scale); each
        // band's total then goes into the row's pair.
        // int8 head: chunk e's two accumulators per column, the offset
        // removed with the chunk's activation sums, the unit's logits written
        // and each warp's best (logit, lowest row) merged into p.keys.
        auto epilogue_i8 = [&](int e) {
            const int eb = e & 1;
            const Item &it = p.item[prev_item];
            const uint32_t *xm = meta_s + kXmWords * eb;
            const int bands = (int)(xm[16] & 3u);
            const int n = mma_n(it.m, bands), cols = n == 32 ? 2 : kCols;
            uint32_t good = 1u;
            if (lane == 0) good = waiter.wait(bars + kBarDFull + 8 * eb, (e >> 1) & 1) ? 1u : 0u;
            good = __shfl_sync(0xFFFFFFFFu, good, 0);
            if (good) {
                ptx::tc_fence_after();
                const uint32_t bl = tmem + ((uint32_t)(quad * 32) << 16) + kDColL + (uint32_t)(n * cols * eb);
                const uint32_t bh = bl + (kDColH - kDColL);
                // per activation row: both nibbles' sums, b = 16 (h - 8) + l,
                // so sum b x = 2^13 sum h' x + 2^9 sum l' x - 128 sum x where
                // h' = h 2^-9 and l' = l 2^-9 are the MMA's A values
                for (int h = 0; h < 2 && 16 * h < 2 * bands * it.m; ++h) {
                    float dl[16], dh[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) dl[q] = dh[q] = 0.f;
                    for (int c = 0; c < cols; ++c) {
                        uint32_t vl[16], vh[16];
                        ptx::tmem_ld_32x32b_x16(bl + (uint32_t)(n * c + 16 * h), vl);
                        ptx::tmem_ld_32x32b_x16(bh + (uint32_t)(n * c + 16 * h), vh);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            dl[q] += __uint_as_float(vl[q]);
                            dh[q] += __uint_as_float(vh[q]);
                        }
                    }
                    if (bands == 1) {  // column 2i: hi, 2i + 1: lo term of row i
#pragma unroll
                        for (int mm = 0; mm < 8; ++mm) {
                            if (mm < it.m) {
                                const int sa = row_scale_exp(xm[2 * mm]);
                                const float fa = exp2i(-sa), fb = exp2i(-sa - 4);
                                acc_pair(acc[mm], acc_lo[mm], 8192.f * fmaf(dh[2 * mm + 1], fb, dh[2 * mm] * fa));
                                acc_pair(acc[mm], acc_lo[mm], 512.f * fmaf(dl[2 * mm + 1], fb, dl[2 * mm] * fa));
                            }
                        }
                    } else {  // column 4i + b: hi_A, lo_A, hi_B, lo_B of row i
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const int mm = 4 * h + r;
                            if (mm < it.m) {
                                const int sa = row_scale_exp(xm[2 * mm]), sb = row_scale_exp(xm[2 * mm + 1]);
                                const float fa = exp2i(-sa), fa4 = exp2i(-sa - 4), fb = exp2i(-sb), fb4 = exp2i(-sb - 4);
                                acc_pair(acc[mm], acc_lo[mm], 8192.f * fmaf(dh[4 * r + 1], fa4, dh[4 * r] * fa));
                                acc_pair(acc[mm], acc_lo[mm], 8192.f * fmaf(dh[4 * r + 3], fb4, dh[4 * r + 2] * fb));
                                acc_pair(acc[mm], acc_lo[mm], 512.f * fmaf(dl[4 * r + 1], fa4, dl[4 * r] * fa));
                                acc_pair(acc[mm], acc_lo[mm], 512.f * fmaf(dl[4 * r + 3], fb4, dl[4 * r + 2] * fb));
                            }
                        }
                    }
                }
#pragma unroll
                for (int mm = 0; mm < 8; ++mm) {
                    if (mm < it.m) {
                        acc_pair(acc[mm], acc_lo[mm], -128.f * __uint_as_float(xm[32 + 2 * mm]));
                        acc_pair(acc[mm], acc_lo[mm], -128.f * __uint_as_float(xm[33 + 2 * mm]));
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bars + kBarDEmpty + 8 * eb);
            if (!prev_last) return;
            const int r = prev_tile * 128 + i;
            const bool live = r < it.rows;
            const float sc = live ? it.scale_g[r] : 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (q < it.m) {
                    float yv = sc * __fadd_rn(acc[q], acc_lo[q]);
                    if (yv == 0.f) yv = 0.f;  // one zero for the order below
                    if (live) it.y[(size_t)q * it.rows + r] = yv;
                    // order-preserving bits of the logit, then the inverted row:
                    // the largest key is the largest logit at the lowest row
                    const uint32_t u = __float_as_uint(yv);
                    const uint32_t ou = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
                    unsigned long long key = live ? ((unsigned long long)ou << 32) | (unsigned long long)(~(uint32_t)r) : 0ull;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, key, o);
                        key = other > key ? other : key;
                    }
                    if (lane == 0 && key != 0ull) atomicMax(p.keys + q, key);
                }
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = acc_lo[q] = 0.f;
        };

        auto epilogue = [&](int e) {
            if constexpr (kI8) {
                epilogue_i8(e);
                return;
            }
            const int eb = e & 1;
            const Item &it = p.item[prev_item];
            const uint32_t *xm = meta_s + kXmWords * eb;
            const int bands = (int)(xm[16] & 3u);
            const int n = mma_n(it.m, bands), cols = n == 32 ? 2 : kCols;
            pairs = pairs || bands == 2;
            uint32_t good = 1u;
            if (lane == 0) good = waiter.wait(bars + kBarDFull + 8 * eb, (e >> 1) & 1) ? 1u : 0u;
            good = __shfl_sync(0xFFFFFFFFu, good, 0);
            // one band: column 2i holds the hi, 2i + 1 the lo terms of row i,
            // summed over the issuing columns here and scaled once D is free
            float dsum[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) dsum[q] = 0.f;
            if (good) {
                ptx::tc_fence_after();
                const uint32_t base = tmem + ((uint32_t)(quad * 32) << 16) + kDCol + (uint32_t)(n * cols * eb);
                if (bands == 1 && it.m == 1) {  // the decode-time GEMV: two live columns of each
                    uint32_t dv[kCols][4];
#pragma unroll
                    for (int c = 0; c < kCols; ++c) ptx::tmem_ld_32x32b_x4(base + 16u * (uint32_t)c, dv[c]);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < kCols; ++c) {
                        dsum[0] += __uint_as_float(dv[c][0]);
                        dsum[1] += __uint_as_float(dv[c][1]);
                    }
                } else if (bands == 1) {
#pragma unroll 1
                    for (int c = 0; c < kCols; ++c) {
                        uint32_t dv[16];
                        ptx::tmem_ld_32x32b_x16(base + 16u * (uint32_t)c, dv);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 16; ++q) dsum[q] += __uint_as_float(dv[q]);
                    }
                } else {
                    // two bands: column 4i + b holds hi_A, lo_A, hi_B, lo_B of
                    // row i, rows 4h .. 4h + 3 in TMEM columns 16h .. 16h + 15
                    // of every issuing column; each band's total goes into
                    // the row's pair
                    for (int h = 0; h < 2 && 16 * h < 4 * it.m; ++h) {
                        float d2[16];
#pragma unroll
                        for (int q = 0; q < 16; ++q) d2[q] = 0.f;
                        for (int c = 0; c < cols; ++c) {
                            uint32_t dv[16];
                            ptx::tmem_ld_32x32b_x16(base + (uint32_t)(n * c + 16 * h), dv);
                            ptx::tmem_wait_ld();
#pragma unroll
                            for (int q = 0; q < 16; ++q) d2[q] += __uint_as_float(dv[q]);
                        }
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const int mm = 4 * h + r;
                            if (mm < it.m) {
                                const int sa = row_scale_exp(xm[2 * mm]), sb = row_scale_exp(xm[2 * mm + 1]);
                                acc_pair(acc[mm], acc_lo[mm],
                                         fmaf(d2[4 * r + 1], exp2i(-sa - 4), d2[4 * r] * exp2i(-sa)));
                                acc_pair(acc[mm], acc_lo[mm],
                                         fmaf(d2[4 * r + 3], exp2i(-sb - 4), d2[4 * r + 2] * exp2i(-sb)));
                            }
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bars + kBarDEmpty + 8 * eb);
            if (good && bands == 1) {
#pragma unroll
                for (int mm = 0; mm < 8; ++mm) {
                    if (mm < it.m) {
                        const int sa = row_scale_exp(xm[2 * mm]);
                        const float t = fmaf(dsum[2 * mm + 1], exp2i(-sa - 4), dsum[2 * mm] * exp2i(-sa));
                        if (pairs)
                            acc_pair(acc[mm], acc_lo[mm], t);
                        else
                            acc[mm] += t;
                    }
                }
            }
            if (!prev_last) return;
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = __fadd_rn(acc[q], acc_lo[q]);
            pairs = false;
            if (it.swiglu) {
                const int r = prev_tile * 64 + (i & 63);
                if (i >= 64 && r < it.rows) {
                    const float su = it.scale_u[r];
#pragma unroll
                    for (int q = 0; q < 8; ++q) xch[(i - 64) * 8 + q] = su * (0.5f * acc[q]);
                }
                ptx::named_bar_sync(1, kStagers);
                if (i < 64 && r < it.rows) {
                    const float sg = it.scale_g[r];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        if (q < it.m) it.y[(size_t)q * it.rows + r] = silu_f(sg * (0.5f * acc[q])) * xch[i * 8 + q];
                }
                ptx::named_bar_sync(1, kStagers);  // xch reusable
            } else {
                const int r = prev_tile * 128 + i;
                if (r < it.rows) {
                    const float sc = it.scale_g[r];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        if (q < it.m) it.y[(size_t)q * it.rows + r] = sc * (0.5f * acc[q]);
                }
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = acc_lo[q] = 0.f;
        };

        // Waits (lane 0 of each staging warp, then the warp) until chunk
        // gc - 1's MMAs are done with the other B buffer: a two-band chunk
        // takes both buffers, and so did a previous two-band chunk.
        auto wait_other_buffer = [&]() {
            if (gc >= 1 && lane == 0)
                waiter.wait(bars + kBarBEmpty + 8 * ((gc - 1) & 1), (uint32_t)((gc - 1) >> 1) & 1u);
            __syncwarp();
        };
        // Two-band operand of a chunk from x in global memory (normalised
        // again with the row's factor for items with a norm), with each
        // row's maxima already in xm (both buffers, from the first; the
        // callers have waited for them).
        auto build_two_band = [&](const Item &it, int w0, int n_words, const uint32_t *xm) {
            const int m = it.m, kw = it.k / 16;
            const uint32_t wbytes = b_block_bytes(m, 2);
#pragma unroll 1
            for (int item = st_tid; item < m * n_words; item += kStagers) {
                const int mm = item / n_words, wi = item - mm * n_words, gw = w0 + wi;
                uint4 va = make_uint4(0u, 0u, 0u, 0u), vb = va;
                if (gw < kw) {
                    const uint4 *xr = reinterpret_cast<const uint4 *>(it.x + (size_t)mm * it.k) + 2 * gw;
                    va = xr[0];
                    vb = xr[1];
                    if (it.norm_w != nullptr)
                        rmsnorm_word(va, vb, reinterpret_cast<const float4 *>(it.norm_w) + 4 * gw,
                                     __uint_as_float(xm[24 + mm]));
                }
                uint4 rows[4];
                split_word2(va, vb, exp2i(row_scale_exp(xm[2 * mm])), exp2i(row_scale_exp(xm[2 * mm + 1])),
                            band_threshold2(xm[2 * mm]), rows, kI8);
                const uint32_t at = bbuf + (uint32_t)wi * wbytes + 64u * (uint32_t)mm;
#pragma unroll
                for (int r = 0; r < 4; ++r) ptx::sts128(at + 16u * (uint32_t)r, rows[r]);
            }
        };

        while (ok) {
            const int buf = gc & 1;
            const Item &it = p.item[cur.item];
            // the MMAs of chunk gc-2 must be done with this B buffer
            if (lane == 0) waiter.wait(bars + kBarBEmpty + 8 * buf, ((gc >> 1) & 1) ^ 1);
            __syncwarp();
            if (prev_bands == 2) wait_other_buffer();
            uint32_t *xm = meta_s + kXmWords * buf;
            const bool reuse = held_item[buf] == cur.item && held_chunk[buf] == cur.chunk;
            // Past this barrier every staging warp has finished chunk gc-2's
            // epilogue, the last reader of this buffer's metadata xm.  The
            // barrier ORs the abort flag over the four staging warps, so they
            // all take the same branch.
            if (ptx::named_bar_or(1, kStagers, *abort_flag != 0u)) break;
            int bands = 1;
            const uint32_t bfull = bars + kBarBFull + 8 * buf;
            if (!reuse) {
                const int m = it.m;
                const int n_words = cur.n_stages_chunk * kSW;
                const int w0 = cur.chunk * cur.cstages * kSW;
                if (it.bsrc != nullptr) {
                    // prepared: the rows' maxima and band-B flags; with one
                    // band the chunk's bytes in a few bulk copies that complete
                    // on BFull (whose phase also waits for every staging
                    // thread's arrival below), with two a build from x here
                    const uint32_t *meta = it.meta + (size_t)kMetaWords * cur.chunk;
                    // each warp reads the rows' flags side by side (one load latency)
                    const uint32_t flag = lane < m ? meta[16 + lane] : 0u;
                    bands = __any_sync(0xFFFFFFFFu, flag != 0u) ? 2 : 1;
                    if (st_tid < 2 * m) xm[st_tid] = meta[st_tid];
                    if (it.norm_w != nullptr && st_tid < m) xm[24 + st_tid] = meta[24 + st_tid];
                    if constexpr (kI8) {
                        if (st_tid < 2 * m) xm[32 + st_tid] = meta[32 + st_tid];
                    }
                    if (bands == 1) {
                        if (st_tid == 0) {
                            const uint32_t bytes = (uint32_t)n_words * b_block_bytes(m, 1);
                            const unsigned char *src = it.bsrc + (size_t)w0 * b_block_bytes(m, 1);
                            const uint32_t bb = bbuf + (uint32_t)buf * kBBufBytes;
                            ptx::mbar_expect_tx(bfull, bytes);
                            for (uint32_t o = 0; o < bytes; o += kBulkPiece)
                                ptx::bulk_load(bb + o, src + o, min(kBulkPiece, bytes - o), bfull);
                        }
                    } else {
                        if (prev_bands != 2) wait_other_buffer();
                        ptx::named_bar_sync(1, kStagers);  // xm complete
                        build_two_band(it, w0, n_words, xm);
                        ptx::fence_proxy_async_smem();  // my B writes -> visible to the tensor core
                    }
                } else {
                    // Built here (m = 1 items).  The row's words are copied
                    // asynchronously into their one-band slots (32 bytes each,
                    // the size of 16 bf16; zero-filled past K); the row
                    // maximum is reduced from shared memory; then each word's
                    // band statistics are taken and the word is split in place
                    // with one band.  If the row needs band B (need_two_bands)
                    // the chunk is built again with two bands from x in
                    // global memory, in both buffers.  A warp's 32 items are
                    // 32 consecutive words of the row.
                    const uint32_t bb = bbuf + (uint32_t)buf * kBBufBytes;
                    float *sabs = reinterpret_cast<float *>(xm + 18);
                    if (st_tid == 0) {
                        xm[0] = xm[1] = xm[17] = 0u;
                        *sabs = 0.f;
                    }
                    for (int wi = st_tid; wi < n_words; wi += kStagers) {
                        const int kk = 16 * (w0 + wi);
                        const bool in_k = kk < it.k;
                        const uint16_t *src = in_k ? it.x + kk : it.x;
                        ptx::cp_async16(bb + 32u * (uint32_t)wi, src, in_k ? 16u : 0u);
                        ptx::cp_async16(bb + 32u * (uint32_t)wi + 16u, src + 8, in_k ? 16u : 0u);
                    }
                    if (it.norm_w != nullptr) {
                        // RMSNorm: the row's mean square from x in global
                        // memory over the whole row (while the copies fly),
                        // then every thread's own words normalised in place
                        const uint4 *xr = reinterpret_cast<const uint4 *>(it.x);
                        const int kw = it.k / 16;
                        double ss = 0.0;
                        for (int w = st_tid; w < kw; w += kStagers) ss += sumsq16(__ldg(xr + 2 * w), __ldg(xr + 2 * w + 1));
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
                        double *ssred = reinterpret_cast<double *>(xch);  // free until this chunk's epilogue
                        if (lane == 0) ssred[quad] = ss;
                        ptx::named_bar_sync(1, kStagers);
                        const float rn = rms_factor(ssred[0] + ssred[1] + ssred[2] + ssred[3], it.k, p.eps);
                        if (st_tid == 0) xm[24] = __float_as_uint(rn);
                        ptx::cp_async_wait_all();
                        const float4 *g4 = reinterpret_cast<const float4 *>(it.norm_w);
                        for (int wi = st_tid; wi < n_words && w0 + wi < kw; wi += kStagers) {
                            const uint32_t at = bb + 32u * (uint32_t)wi;
                            uint4 va = ptx::lds128(at), vb = ptx::lds128(at + 16u);
                            rmsnorm_word(va, vb, g4 + 4 * (w0 + wi), rn);
                            ptx::sts128(at, va);
                            ptx::sts128(at + 16u, vb);
                        }
                    }
                    ptx::cp_async_wait_all();
                    ptx::named_bar_sync(1, kStagers);
                    double sx = 0.0;  // int8 head: the chunk's activation sum
                    // (every staging thread takes the same number of turns
                    // through the loops with warp reductions: a chunk's word
                    // count need not be a multiple of 32; past it, zeros)
                    for (int base = 0; base < n_words; base += kStagers) {
                        const int wi = base + st_tid;
                        const uint32_t at = bb + 32u * (uint32_t)wi;
                        const bool in = wi < n_words;
                        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                        const uint4 va = in ? ptx::lds128(at) : z, vb = in ? ptx::lds128(at + 16u) : z;
                        const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, max_abs16(va, vb));
                        if (lane == 0) atomicMax(&xm[0], mx);
                        if constexpr (kI8) sx += sum16(va, vb);
                    }
                    if constexpr (kI8) {
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) sx += __shfl_xor_sync(0xFFFFFFFFu, sx, o);
                        if (lane == 0) reinterpret_cast<double *>(xch)[4 + quad] = sx;
                    }
                    ptx::named_bar_sync(1, kStagers);
                    if constexpr (kI8) {
                        if (st_tid == 0) {
                            const double *d = reinterpret_cast<const double *>(xch) + 4;
                            const double t = d[0] + d[1] + d[2] + d[3];
                            const float hi = (float)t;
                            xm[32] = __float_as_uint(hi);
                            xm[33] = __float_as_uint((float)(t - (double)hi));
                        }
                    }
                    const uint32_t tb2 = band_threshold2(xm[0]);
                    const float sca = exp2i(row_scale_exp(xm[0]));
                    for (int base = 0; base < n_words; base += kStagers) {
                        const int wi = base + st_tid;
                        const uint32_t at = bb + 32u * (uint32_t)wi;
                        const bool in = wi < n_words;
                        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                        const uint4 va = in ? ptx::lds128(at) : z, vb = in ? ptx::lds128(at + 16u) : z;
                        uint32_t cnt = 0;
                        float sa = 0.f;
                        band_stats16(va, vb, tb2, cnt, sa);
                        const uint32_t mb = __reduce_max_sync(0xFFFFFFFFu, max_abs16_below(va, vb, tb2));
                        cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) sa += __shfl_xor_sync(0xFFFFFFFFu, sa, o);
                        if (lane == 0) {
                            atomicMax(&xm[1], mb);
                            atomicAdd(&xm[17], cnt);
                            atomicAdd(sabs, sa);
                        }
                        if (in) {
                            uint4 rows[2];
                            split_word1(va, vb, sca, rows, kI8);
                            ptx::sts128(at, rows[0]);
                            ptx::sts128(at + 16u, rows[1]);
                        }
                    }
                    ptx::named_bar_sync(1, kStagers);
                    bands = need_two_bands(xm[0], xm[17], *sabs) ? 2 : 1;
                    if (bands == 2) {
                        if (prev_bands != 2) wait_other_buffer();
                        ptx::named_bar_sync(1, kStagers);  // both buffers are free
                        build_two_band(it, w0, n_words, xm);
                    }
                    ptx::fence_proxy_async_smem();  // my B writes -> visible to the tensor core
                }
                if (st_tid == 0) xm[16] = ((uint32_t)gc << 2) | (uint32_t)bands;
                if (bands == 2) {  // both buffers are overwritten: neither holds a reusable chunk
                    held_item[0] = held_item[1] = -1;
                } else {
                    held_item[buf] = cur.item;
                    held_chunk[buf] = cur.chunk;
                }
            } else if (st_tid == 0) {
                xm[16] = ((uint32_t)gc << 2) | 1u;  // the same one-band chunk again, under this chunk's number
            }
            last_gc[buf] = gc;
            ptx::mbar_arrive(bfull);
            if (gc >= 1) epilogue(gc - 1);
            prev_item = cur.item;
            prev_tile = cur.tile;
            prev_last = cur.last_chunk_of_unit();
            prev_bands = bands;
            ++gc;
            ok = cur.next_chunk();
        }
        if (!ptx::named_bar_or(1, kStagers, *abort_flag != 0u) && gc >= 1) epilogue(gc - 1);
        // After an abort a bulk copy into a B buffer may still be in flight:
        // its buffer's last BFull phase completes only when it has landed
        // (every staging thread has arrived on it).
        if (st_tid == 0)
            for (int b = 0; b < 2; ++b)
                if (last_gc[b] >= 0)
                    drain_wait(bars + kBarBFull + 8 * b, (uint32_t)(last_gc[b] >> 1) & 1u, &g_batched_error);
    }

    __syncthreads();
    if (warp == 0) {
        // every MMA of this CTA has completed before its tensor memory is released
        if (lane == 0) drain_wait(bars + kBarDrain, 0, &g_batched_error);
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// Launch groups of a batch: consecutive runs of items, each with up to
// kMaxItems items that have rows > 0 and k > 0 ("real" items) holding up to
// kMaxMaps tensor maps.  The fewest groups a greedy walk needs is found
// first, then the real items are spread evenly over that many groups (a
// short last launch streams far below the rate of a full one).  Items with
// rows == 0 (nothing to do) or k == 0 (y = 0, written by a small CUDA-core
// launch of their own) ride along without counting.  Returns the end index of
// each group.
std::vector<int> plan_groups(const tern_batch_item *items, int n)
{
    auto walk = [&](int per_group) {
        std::vector<int> ends;
        int cnt = 0, n_maps = 0;
        for (int idx = 0; idx < n; ++idx) {
            const tern_batch_item &b = items[idx];
            if (b.w->rows == 0 || b.w->k == 0) continue;
            const int need = b.up ? 2 : 1;
            if (cnt == per_group || n_maps + need > kMaxMaps) {
                ends.push_back(idx);
                cnt = 0;
                n_maps = 0;
            }
            ++cnt;
            n_maps += need;
        }
        ends.push_back(n);
        return ends;
    };
    int real = 0;
    for (int idx = 0; idx < n; ++idx) real += (items[idx].w->rows != 0 && items[idx].w->k != 0) ? 1 : 0;
    const std::vector<int> greedy = walk(kMaxItems);
    if (greedy.size() <= 1) return greedy;
    const int per = (real + (int)greedy.size() - 1) / (int)greedy.size();
    std::vector<int> even = walk(per);
    return even.size() <= greedy.size() ? even : greedy;
}

// Workspace of prepared activations per (context, stream), grown on demand.
// A grown-out buffer is never freed: a launch captured in a CUDA graph keeps
// the address it was captured with.  Returns nullptr if the allocation fails
// (the call then returns TERN_ERR_CUDA; the groups before it have launched).
void *workspace(cudaStream_t stream, size_t need, int slot = 0)
{
    struct Buf {
        void *p = nullptr;
        size_t bytes = 0;
    };
    static std::mutex mu;
    static std::map<std::pair<unsigned long long, cudaStream_t>, Buf> all_slots[2];  // 0: prepared B, 1: head keys
    auto &all = all_slots[slot];
    // keyed by the current context: a context created after a device reset
    // gets buffers of its own
    const unsigned long long ctx = current_context_id();
    if (ctx == 0) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    Buf &b = all[{ctx, stream}];
    if (b.bytes >= need) return b.p;
    const size_t bytes = need > 2 * b.bytes ? need : 2 * b.bytes;
    // an allocation is allowed while a stream of this thread is being captured
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    if (cudaThreadExchangeStreamCaptureMode(&mode) != cudaSuccess) return nullptr;
    void *p = nullptr;
    const cudaError_t e = cudaMalloc(&p, bytes);
    cudaThreadExchangeStreamCaptureMode(&mode);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    b.p = p;
    b.bytes = bytes;
    return p;
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// 512-code stages over K, and stages per chunk: the fewest chunks that fit a
// B buffer, of equal stage counts (a short last chunk would pay the
// per-chunk costs for little work).
void chunk_plan(int k, int m, int &stages, int &cstages, int sw = kStageWords)
{
    stages = (k / 16 + sw - 1) / sw;
    const int cap = kBBufBytes / (sw * (int)b_block_bytes(m, 1));  // stages of one-band B one buffer holds
    const int n_chunks = (stages + cap - 1) / cap;
    cstages = (stages + n_chunks - 1) / n_chunks;
}

// Workspace bytes of one prepared item (see Item::bsrc, Item::meta).
size_t prep_b_bytes(int stages, int m, int sw = kStageWords)
{
    return align256((size_t)stages * sw * b_block_bytes(m, 1));
}
size_t prep_bytes(int stages, int cstages, int m, int sw = kStageWords)
{
    const int n_chunks = (stages + cstages - 1) / cstages;
    return prep_b_bytes(stages, m, sw) + align256((size_t)n_chunks * kMetaWords * sizeof(uint32_t));
}

// Scratch of tern_gemm_batched_noalloc: module-scope device memory, which the
// CUDA runtime sets up when it loads the library's kernels on a device, so
// the entry point itself never allocates.
__device__ __align__(256) unsigned char g_noalloc_ws[TERN_NOALLOC_WS_BYTES];

}  // namespace

int batched_launches(const tern_batch_item *items, int n)
{
    int launches = 0, begin = 0;
    for (const int end : plan_groups(items, n)) {
        bool any = false, prep = false;
        for (int i = begin; i < end; ++i) {
            if (items[i].w->rows == 0) continue;
            if (items[i].w->k == 0) {
                ++launches;
            } else {
                any = true;
                prep = prep || items[i].m >= 2;
            }
        }
        launches += (any ? 1 : 0) + (prep ? 1 : 0);
        begin = end;
    }
    return launches;
}

namespace {

// One product of a launch group, in the form the launch needs.  codes_*:
// the weights as uint32 words, kw per row (16 ternary codes or 4 int8
// weights a word).
struct Job {
    const uint32_t *codes_g, *codes_u;  // codes_u: the up projection of a SwiGLU pair, or nullptr
    const float *scale_g, *scale_u;
    const uint16_t *x;
    float *y;
    const float *norm_w;
    int rows, k, m, kw;
};

// Launches one group (cnt jobs, each with rows > 0 and k > 0): the preparing
// kernel if some job has m >= 2, then the persistent kernel of format kFmt.
// fixed_ws: a workspace the caller guarantees to be large enough (nullptr:
// the per-stream workspace).  keys: the int8 head's argmax keys.
template <int kFmt>
tern_status launch_group(const Job *jobs, int cnt, cudaStream_t stream, unsigned char *fixed_ws, float eps,
                         unsigned long long *keys)
{
    static_assert(sizeof(Params) + sizeof(Maps) < 32000, "kernel parameters exceed 32 KB");
    constexpr int kSW = stage_b_words(kFmt);
    const int sms = sm_count();
    // the kernel's shared-memory attribute, once per context (a context
    // created after a device reset starts without it)
    {
        static std::mutex mu;
        static std::set<unsigned long long> done;
        const unsigned long long ctx = current_context_id();
        std::lock_guard<std::mutex> lock(mu);
        if (ctx == 0 || done.count(ctx) == 0) {
            if (cudaFuncSetAttribute(k_tern_batched<kFmt>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemBytes) != cudaSuccess)
                return TERN_ERR_CUDA;
            if (ctx != 0) done.insert(ctx);
        }
    }
    Params prm;
    std::memset(&prm, 0, sizeof(prm));
    Maps maps;
    std::memset(&maps, 0, sizeof(maps));
    std::vector<long long> unit_cost;
    int units = 0, n_maps = 0;
    for (int j = 0; j < cnt; ++j) {
        const Job &b = jobs[j];
        Item &it = prm.item[j];
        it.scale_g = b.scale_g;
        it.scale_u = b.scale_u;
        it.x = b.x;
        it.y = b.y;
        it.rows = b.rows;
        it.k = b.k;
        it.m = b.m;
        it.swiglu = b.codes_u != nullptr;
        it.norm_w = b.norm_w;
        chunk_plan(it.k, it.m, it.stages, it.cstages, kSW);
        it.unit0 = units;
        it.map = n_maps;
        const int tile_rows = it.swiglu ? 64 : 128;
        const int tiles = (it.rows + tile_rows - 1) / tile_rows;
        if (!make_code_map(&maps.m[n_maps++], b.codes_g, it.rows, b.kw, tile_rows)) return TERN_ERR_CUDA;
        if (it.swiglu && !make_code_map(&maps.m[n_maps++], b.codes_u, it.rows, b.kw, tile_rows))
            return TERN_ERR_CUDA;
        for (int t = 0; t < tiles; ++t) unit_cost.push_back(it.stages);
        units += tiles;
    }
    prm.n_items = cnt;
    prm.eps = eps;
    prm.wait_limit = wait_limit();
    prm.keys = keys;

    // Items with m >= 2 take their B from the workspace, written by one
    // k_tern_bprep launch just before (one CTA per item, K chunk and
    // activation row): per item the padded K's one-band words (32m bytes
    // per 16 activations), then kMetaWords of metadata per chunk.  Items
    // with m = 1 are built by the persistent kernel's staging warps.
    PrepParams pp;
    std::memset(&pp, 0, sizeof(pp));
    pp.eps = eps;
    size_t ws_need = 0;
    std::vector<std::pair<size_t, size_t>> ws_off(cnt);
    for (int j = 0; j < cnt; ++j) {
        const Item &it = prm.item[j];
        if (it.m < 2) continue;
        ws_off[j].first = ws_need;
        ws_off[j].second = ws_need + prep_b_bytes(it.stages, it.m, kSW);
        ws_need += prep_bytes(it.stages, it.cstages, it.m, kSW);
    }
    if (ws_need > 0) {
        unsigned char *ws = fixed_ws != nullptr ? fixed_ws : static_cast<unsigned char *>(workspace(stream, ws_need));
        if (ws == nullptr) return TERN_ERR_CUDA;
        for (int j = 0; j < cnt; ++j) {
            Item &it = prm.item[j];
            if (it.m < 2) continue;
            it.bsrc = ws + ws_off[j].first;
            it.meta = reinterpret_cast<const uint32_t *>(ws + ws_off[j].second);
            PrepItem &q = pp.item[pp.n_items++];
            q.x = it.x;
            q.norm_w = it.norm_w;
            q.sw = kSW;
            q.head = kFmt == kFmtI8 ? 1 : 0;
            q.b = ws + ws_off[j].first;
            q.meta = reinterpret_cast<uint32_t *>(ws + ws_off[j].second);
            q.k = it.k;
            q.m = it.m;
            q.stages = it.stages;
            q.cstages = it.cstages;
            q.task0 = pp.n_tasks;
            if (it.cstages * kSW > kPrepWords * kPrepThreads) return TERN_ERR_SHAPE;  // cannot happen: m >= 2
            pp.n_tasks += (it.stages + it.cstages - 1) / it.cstages * it.m;
        }
        cudaLaunchConfig_t pcfg = {};
        pcfg.gridDim = dim3((unsigned)pp.n_tasks, 1, 1);
        pcfg.blockDim = dim3(kPrepThreads, 1, 1);
        pcfg.stream = stream;
        cudaLaunchAttribute pattr;
        pattr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pattr.val.programmaticStreamSerializationAllowed = 1;
        pcfg.attrs = &pattr;
        pcfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&pcfg, k_tern_bprep, pp) != cudaSuccess) return TERN_ERR_CUDA;
    }
    // contiguous runs of units with balanced stage counts
    const int ctas = units < sms ? units : (sms < kMaxCtas ? sms : kMaxCtas);
    long long total = 0;
    for (long long c : unit_cost) total += c;
    int u = 0;
    long long acc = 0;
    prm.unit_start[0] = 0;
    for (int b = 1; b < ctas; ++b) {
        const long long target = total * b / ctas;
        while (u < units && acc + unit_cost[u] / 2 < target) acc += unit_cost[u++];
        prm.unit_start[b] = u;
    }
    prm.unit_start[ctas] = units;
    for (int b = 0, j = 0; b < ctas; ++b) {
        while (j + 1 < cnt && prm.item[j + 1].unit0 <= prm.unit_start[b]) ++j;
        prm.item_start[b] = j;
    }
    for (int b = 0; b < ctas; ++b) {
        long long st = 0;
        for (int q = prm.unit_start[b]; q < prm.unit_start[b + 1]; ++q) st += unit_cost[q];
        prm.stages_cta[b] = (int)st;
    }

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k_tern_batched<kFmt>, prm, maps) != cudaSuccess) return TERN_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return TERN_ERR_CUDA;
    return TERN_OK;
}

// Launches the batch, group by group.  fixed_ws: see launch_group.  norm_w:
// nullptr, or per item the RMSNorm channel weights (nullptr for an item
// without a norm), with eps.
tern_status run_batched(const tern_batch_item *items, int n, cudaStream_t stream, unsigned char *fixed_ws,
                        const float *const *norm_w = nullptr, float eps = 0.f)
{
    int begin = 0;
    std::vector<Job> jobs;
    for (const int end : plan_groups(items, n)) {
        jobs.clear();
        for (int idx = begin; idx < end; ++idx) {
            const tern_batch_item &b = items[idx];
            if (b.w->rows == 0) continue;
            if (b.w->k == 0) {  // empty sum: y = scale * 0
                const tern_status st = empty_sum(b.w, b.up, b.m, b.y, stream);
                if (st != TERN_OK) return st;
                continue;
            }
            Job jb;
            jb.codes_g = b.w->codes;
            jb.codes_u = b.up ? b.up->codes : nullptr;
            jb.scale_g = b.w->scale;
            jb.scale_u = b.up ? b.up->scale : nullptr;
            jb.x = b.x;
            jb.y = b.y;
            jb.norm_w = norm_w != nullptr ? norm_w[idx] : nullptr;
            jb.rows = b.w->rows;
            jb.k = b.w->k;
            jb.m = b.m;
            jb.kw = b.w->k / 16;
            jobs.push_back(jb);
        }
        begin = end;
        if (jobs.empty()) continue;
        const tern_status st = launch_group<kFmtTern>(jobs.data(), (int)jobs.size(), stream, fixed_ws, eps, nullptr);
        if (st != TERN_OK) return st;
    }
    return TERN_OK;
}

// The int8 head's argmax keys start below every real key (a real key's top
// half is the order-preserving image of a finite logit, never zero).
__global__ void k_head_keys_init(unsigned long long *keys)
{
    if (threadIdx.x < 8) keys[threadIdx.x] = 0ull;
}

// The int8 head's argmax: the key of each activation row back to its row.
__global__ void k_head_argmax_finish(const unsigned long long *keys, int32_t *argmax, int m)
{
    const int q = (int)threadIdx.x;
    if (q < m) argmax[q] = (int32_t)(~(uint32_t)(keys[q] & 0xFFFFFFFFull));
}

}  // namespace

tern_status gemm_batched(const tern_batch_item *items, int n, cudaStream_t stream)
{
    return run_batched(items, n, stream, nullptr);
}

tern_status gemm_batched_rmsnorm(const tern_batch_item *items, const float *const *norm_w, float eps, int n,
                                 cudaStream_t stream)
{
    return run_batched(items, n, stream, nullptr, norm_w, eps);
}

tern_status head_argmax(const tern_i8_matrix *w, const uint16_t *x, int m, const float *norm_w, float eps,
                        float *logits, int32_t *argmax, cudaStream_t stream)
{
    unsigned long long *keys = static_cast<unsigned long long *>(workspace(stream, 8 * sizeof(unsigned long long), 1));
    if (keys == nullptr) return TERN_ERR_CUDA;
    Job jb;
    jb.codes_g = reinterpret_cast<const uint32_t *>(w->w);
    jb.codes_u = nullptr;
    jb.scale_g = w->scale;
    jb.scale_u = nullptr;
    jb.x = x;
    jb.y = logits;
    jb.norm_w = norm_w;
    jb.rows = w->rows;
    jb.k = w->k;
    jb.m = m;
    jb.kw = w->k / 4;
    k_head_keys_init<<<1, 32, 0, stream>>>(keys);
    if (cudaGetLastError() != cudaSuccess) return TERN_ERR_CUDA;
    const tern_status st = launch_group<kFmtI8>(&jb, 1, stream, nullptr, eps, keys);
    if (st != TERN_OK) return st;
    k_head_argmax_finish<<<1, 32, 0, stream>>>(keys, argmax, m);
    return cudaGetLastError() == cudaSuccess ? TERN_OK : TERN_ERR_CUDA;
}

tern_status gemm_batched_noalloc(const tern_batch_item *items, int n, cudaStream_t stream)
{
    // every launch group's prepared activations must fit the static scratch
    // (the groups run one after another on the stream and reuse it)
    int begin = 0;
    for (const int end : plan_groups(items, n)) {
        size_t need = 0;
        for (int i = begin; i < end; ++i) {
            const tern_batch_item &b = items[i];
            if (b.w->rows == 0 || b.w->k == 0 || b.m < 2) continue;
            int stages = 0, cstages = 0;
            chunk_plan(b.w->k, b.m, stages, cstages);
            need += prep_bytes(stages, cstages, b.m);
        }
        if (need > (size_t)TERN_NOALLOC_WS_BYTES) return TERN_ERR_SHAPE;
        begin = end;
    }
    // The scratch's device address, looked up with the device current the
    // first time a context uses this entry point.  The cache is keyed by the
    // context, so a context created after a device reset (whose module, and
    // array, are new) looks the address up again.
    static std::mutex mu;
    static std::map<unsigned long long, void *> addr;
    const unsigned long long ctx = current_context_id();
    void *ws = nullptr;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto f = ctx != 0 ? addr.find(ctx) : addr.end();
        if (f != addr.end()) {
            ws = f->second;
        } else {
            if (cudaGetSymbolAddress(&ws, g_noalloc_ws) != cudaSuccess || ws == nullptr) {
                (void)cudaGetLastError();
                return TERN_ERR_CUDA;
            }
            if (ctx != 0) addr[ctx] = ws;
        }
    }
    return run_batched(items, n, stream, static_cast<unsigned char *>(ws));
}

tern_status take_batched_error()
{
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_batched_error, sizeof(v)) != cudaSuccess) return TERN_ERR_CUDA;
    if (v != 0u) {
        if (cudaMemcpyToSymbol(g_batched_error, &z, sizeof(z)) != cudaSuccess) return TERN_ERR_CUDA;
        return TERN_ERR_TIMEOUT;
    }
    return TERN_OK;
}

}  // namespace tern
