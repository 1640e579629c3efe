// compress.cu -- dgc_compress, dgc_compress_shared: the DGC per-worker compressor on sm_103a.
//
// Sources: "[Paper Review] Deep Gradient Compression: Reducing the Communication Bandwidth for
// Distributed Training" (Abstract; Proposed method bullets 1, 3, 4, 5; Research questions RQ4),
// "AdaComp : Adaptive Residual Gradient Compression for Data-Parallel Distributed Training"
// (abstract; citation snippets on magnitude and bin-local selection) and the ScaleComp abstract
// (low-pass filter in the local accumulation; one index set for all learners).
//
// One dgc_compress call enqueues this pipeline on the caller's stream (every kernel reads the
// segment table and counters the previous ones left in the workspace, so no host round trip):
//
//   plan          segment table: k, sample counts, seeds, bins; validates seg_off; zeroes counters
//   clip_tiles    [clipping] exact sum of g^2 per segment in integer arithmetic (a 128-bit
//                 window per thread, 640-bit sums per segment); the block finishing a
//                 segment's last tile rounds it once to binary64 -> scale
//   cache         [sampled, exact] the sample positions, kept sorted in the workspace; checked
//                 every call (tag + checksum), rebuilt only when they no longer match (one
//                 cooperative launch)
//   sample        gathers g,u,v at the SplitMix64 sample positions, recomputes v' there,
//                 writes the sample keys and the first radix-select histogram
//   select x2     radix select of the sampled threshold t (11 + 10 + 10 key bits): segments
//                 whose sample fits on chip in one block each, the rest by the cooperative
//                 global-memory select (one launch, grid barriers between levels)
//   stream_tma    THE STREAMING PASS: persistent blocks, bulk-copy pipeline of g,u,v tiles;
//                 u = fma(m,u,g*scale); v = fma(leak,v,u); candidates (key(v) >= t, or for
//                 AdaComp the entries at their bin run's maximum, which also raise the bin's
//                 global maximum) are compacted into each tile's own slots
//   collect(+copy) tile slots -> one index-ordered candidate list (decoupled look-back)
//   candoff       per-segment candidate ranges; decides who re-selects
//   recompact     [exact mode, only if the sampled bound was too tight] re-compacts from v
//   cval          every candidate's value, gathered once by the whole grid
//   select x2     radix select of the exact k-th (|v|, index) pair among candidates (on chip,
//                 then the global-memory levels for larger candidate sets)
//   emit          writes S in index order (second look-back), clears v (and u with masking)
//                 of the sent entries; statistics
//
// Exact mode uses the sampled threshold only as a safe lower bound: a margin above the sample
// rank makes |C| >= k overwhelmingly likely, and when it is not, recompact re-reads v with a
// zero threshold for that segment. Either way S is the exact top-k.
//
// dgc_compress_shared (one index set given by the caller) runs plan, a check of the set,
// clipping, the streaming pass without candidates, and a gather of v at the set.
#include <cmath>
#include <cstring>
#include <type_traits>

#include "dgc_device.cuh"

namespace dgc {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 8;                          // float4 rows per thread in re-compaction
constexpr int kTile = kThreads * kRows * 4;       // 8192 entries per re-compaction tile
// streaming pass shape: entries per tile, tiles in flight per block, blocks per SM. The DGC
// and shared-set passes run 2048 entries x 4 stages x 2 blocks per SM, the AdaComp pass (46%
// more instructions per entry) 3 stages x 3 blocks, so that more warps hide its latency: the
// fastest of the shapes measured on GB300 for each.
#ifndef DGC_STREAM_TILE
#define DGC_STREAM_TILE 2048
#endif
#ifndef DGC_STREAM_STAGES
#define DGC_STREAM_STAGES 4
#endif
#ifndef DGC_STREAM_BLOCKS_PER_SM
#define DGC_STREAM_BLOCKS_PER_SM 2
#endif
#ifndef DGC_ADACOMP_STAGES
#define DGC_ADACOMP_STAGES 3
#endif
#ifndef DGC_ADACOMP_BLOCKS_PER_SM
#define DGC_ADACOMP_BLOCKS_PER_SM 3
#endif
constexpr int kPTile = DGC_STREAM_TILE;
template <int kSel>
__host__ __device__ constexpr int stream_stages() {
    return kSel == 1 ? DGC_ADACOMP_STAGES : DGC_STREAM_STAGES;
}
template <int kSel>
__host__ __device__ constexpr int stream_blocks_per_sm() {
    return kSel == 1 ? DGC_ADACOMP_BLOCKS_PER_SM : DGC_STREAM_BLOCKS_PER_SM;
}
constexpr int kPRows = kPTile / (4 * kThreads);   // float4 rows per thread
constexpr int kWarps = kThreads / 32;
static_assert(kPRows >= 1 && kPRows * 4 * kThreads == kPTile, "tile = rows x 1024 entries");
static_assert(kPRows * kWarps <= 32, "one warp scans the per-(row, warp) counts");
// the AdaComp pass finds bins with (x + 0.5) * fl(1/L) for x < L + kPTile, L < kPTile: equal to
// x / L for every L in [4, 4095] and x < L + 4096, checked exhaustively in binary32 on the host
// by tests/test_adacomp_bin_index_host.py
static_assert(kPTile <= 4096, "bin index by reciprocal is only checked up to 4096-entry tiles");
constexpr uint32_t kPStageFloats = 3u * kPTile;   // g, u, v
template <int kSel>
constexpr size_t stream_smem_bytes() {  // 96 KiB (72 KiB for AdaComp)
    return sizeof(float) * kPStageFloats * stream_stages<kSel>();
}
constexpr uint32_t kMbarSpinLimit = 1u << 22;
constexpr int kEmitRows = 4;
constexpr int kEmitTile = kThreads * kEmitRows * 4;  // 4096 candidates per emit tile
constexpr int kClipTile = 4096;
constexpr int kSqLimbs = 10;   // 640-bit exact sum of squares, 64-bit limbs (when rounded)
constexpr int kSqDigits = 20;  // the same sum as 32-bit digits, each in a 64-bit word
constexpr int kSqWords = kSqDigits + 1;  // + one word of flags (2: +inf seen, 4: NaN seen)
constexpr int kHistBins = 2048;
// DGC pass: a streaming tile with at most this many candidates stores them as sent (v, and u with
// masking, zeroed) and keeps their values in its slots; the emit step puts back the unsent ones
constexpr uint32_t kSpecSlots = 64;
constexpr uint64_t kExactSamplePpb = 10000000;    // exact mode samples 1% to bound t from below
constexpr uint32_t kExactWholeBelow = 8192;       // smaller segments: every entry is a candidate

// composite selection key X = (|v| key << 32) | ~index, selected from the top 11+10+10 key
// bits then 11+11+10 index bits
__constant__ int c_shift[6] = {52, 42, 32, 21, 10, 0};
__constant__ int c_bits[6] = {11, 10, 10, 11, 11, 10};

enum : uint32_t { kIdle = 0, kActive = 1 };

struct SegInfo {
    uint64_t seed;      // per-segment SplitMix64 seed
    uint64_t prefix;    // radix-select prefix found so far
    uint64_t sel_x;     // selected <=> X >= sel_x
    uint32_t start, end;
    uint32_t k;         // target count
    uint32_t ms;        // sample draws (0: no sampling)
    uint32_t rank;      // rank of the threshold among the samples
    uint32_t thresh;    // candidate threshold key (kNoKey: none)
    uint32_t need;      // radix select: items still to take
    uint32_t state;     // kIdle / kActive
    uint32_t cand_cnt;
    uint32_t failed;    // exact mode: fewer candidates than k
    uint32_t resel;     // sampled mode: re-selection ran
    uint32_t min_key;
    float scale;
    uint32_t bbase;     // first position bucket of the segment
    uint32_t binbase;   // AdaComp: first bin of the segment
    uint32_t nsent;     // AdaComp: entries sent
    double sumsq;       // clipping: S, the squared norm (0 without clipping)
};

struct Ctl {
    int32_t abort;
    uint32_t active;
    uint32_t any_failed;
    uint32_t ticket_fused, ticket_compact, ticket_emit, ticket_collect;
    uint32_t ndense;        // tiles whose slots k_collect_copy moves: up to kCollectWarp ...
    uint32_t nlarge;        // ... and more (listed from the end of dlist)
    uint32_t total_samples, total_clip_tiles, total_cand, total_sent;
    uint32_t emit_done;
    uint64_t tag;           // what the sample positions depend on, for this call
    uint64_t csum;          // checksum of the cached positions as found
    uint64_t newsum;        // checksum of the rebuilt positions
    uint32_t ncomp;         // sample keys kept by the sample select's second level
    uint32_t bar_count;     // grid barrier of the cooperative select: arrivals, generation
    uint32_t bar_gen;
    uint32_t unspec;        // the speculative zeros were undone (exact mode's re-compaction)
};

// Header of the sample-position cache kept in the workspace between calls.
struct SampleCache {
    uint64_t magic, tag, checksum, pad;
};
constexpr uint64_t kCacheMagic = 0x53504F5343414348ull;
constexpr int kBucketShift = 10;  // cache order: 1024-entry buckets, segment by segment

// Workspace layout (host computes it; every piece 256-byte aligned).
struct Layout {
    size_t ctl, scache, segs, seg_start, samp_off, clip_off, cand_off, clip_acc, skeys, spos,
        bcount, histA, histB;
    size_t st_collect, st_compact, st_emit, cidx, sidx, sval, su, tcount, tseg, eseg, clip_cnt,
        dlist, binmax, total;
    uint64_t max_samples, max_clip_tiles, fused_tiles, emit_tiles, ptiles, cgroups, nbuckets,
        max_bins;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct HostParams {
    uint32_t mode, mask, clip_on, bin;
    uint64_t d_ppb, r_ppb, q_ppb;
    float momentum, clip_norm;
    uint64_t seed;
    float bin_inv;  // AdaComp: 1/bin rounded to binary32 (used while bin < the tile length)
    float leak;     // v <- fma(leak, v, u); 1 is the plain sum
    uint32_t nospec;  // no speculative sends (a caller-given index set: no candidates)
};

int check_params(const dgc_params* p, HostParams* hp) {
    if (!p) return DGC_EINVAL;
    if (p->mode != DGC_SELECT_EXACT && p->mode != DGC_SELECT_SAMPLED &&
        p->mode != DGC_SELECT_ADACOMP)
        return DGC_EINVAL;
    if (p->mode == DGC_SELECT_ADACOMP && p->bin_size == 0) return DGC_EINVAL;
    hp->bin = p->mode == DGC_SELECT_ADACOMP ? p->bin_size : 0;
    hp->bin_inv = hp->bin ? 1.0f / (float)hp->bin : 0.0f;
    if (!(p->sparsity >= 0.0 && p->sparsity <= 1.0)) return DGC_EINVAL;
    if (!std::isfinite(p->momentum)) return DGC_EINVAL;
    if (std::isnan(p->clip_norm)) return DGC_EINVAL;
    if (!(p->leak >= 0.0f && p->leak <= 1.0f)) return DGC_EINVAL;
    hp->leak = p->leak == 0.0f ? 1.0f : p->leak;  // 0: no filter
    hp->nospec = 0;
    hp->mode = p->mode;
    hp->mask = (p->flags & DGC_FLAG_MASK_MOMENTUM) ? 1u : 0u;
    hp->clip_on = (p->clip_norm > 0.0f && !std::isinf(p->clip_norm)) ? 1u : 0u;
    hp->d_ppb = (uint64_t)llround((1.0 - p->sparsity) * 1e9);
    hp->momentum = p->momentum;
    hp->clip_norm = p->clip_norm;
    hp->seed = p->seed;
    if (p->mode == DGC_SELECT_SAMPLED) {
        if (!(p->sample_ratio > 0.0 && p->sample_ratio <= 1.0)) return DGC_EINVAL;
        hp->r_ppb = (uint64_t)llround(p->sample_ratio * 1e9);
        if (hp->r_ppb == 0) return DGC_EINVAL;
        if (!(p->reselect_factor >= 1.0 && p->reselect_factor <= 16.0)) return DGC_EINVAL;
        hp->q_ppb = (uint64_t)llround(p->reselect_factor * 1e9);
    } else if (p->mode == DGC_SELECT_EXACT) {
        hp->r_ppb = kExactSamplePpb;
        hp->q_ppb = 0;
    } else {  // AdaComp: no sample, no re-selection
        hp->r_ppb = 0;
        hp->q_ppb = 0;
    }
    return DGC_OK;
}

Layout make_layout(int64_t n, int32_t nseg, const HostParams& hp) {
    Layout L{};
    const uint64_t un = (uint64_t)n;
    L.max_samples = count_ppb(un, hp.r_ppb) + (uint64_t)nseg;
    L.max_clip_tiles = hp.clip_on ? (un + kClipTile - 1) / kClipTile + (uint64_t)nseg : 0;
    L.fused_tiles = (un + kTile - 1) / kTile;
    L.ptiles = (un + kPTile - 1) / kPTile;
    L.cgroups = (L.ptiles + kThreads - 1) / kThreads;
    L.nbuckets = (un >> kBucketShift) + 2 * (uint64_t)nseg + 1;  // >= sum of per-segment buckets
    L.max_bins = hp.bin ? un / hp.bin + (uint64_t)nseg + 1 : 0;  // >= sum of per-segment bins
    L.emit_tiles = (un + kEmitTile - 1) / kEmitTile;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align256(o + bytes); return at; };
    L.ctl = take(sizeof(Ctl));
    L.scache = take(sizeof(SampleCache));
    L.segs = take(sizeof(SegInfo) * (size_t)nseg);
    L.seg_start = take(sizeof(uint32_t) * (size_t)(nseg + 1));
    L.samp_off = take(sizeof(uint32_t) * (size_t)(nseg + 1));
    L.clip_off = take(sizeof(uint32_t) * (size_t)(nseg + 1));
    L.cand_off = take(sizeof(uint32_t) * (size_t)(nseg + 1));
    L.clip_acc = take(sizeof(uint64_t) * kSqWords * (size_t)(hp.clip_on ? nseg : 0));
    L.skeys = take(sizeof(uint32_t) * (size_t)L.max_samples);
    L.spos = take(sizeof(uint32_t) * (size_t)L.max_samples);
    L.bcount = take(sizeof(uint32_t) * (size_t)L.nbuckets);
    L.histA = take(sizeof(uint32_t) * (size_t)nseg * kHistBins);
    L.histB = take(sizeof(uint32_t) * (size_t)nseg * kHistBins);
    L.st_collect = take(sizeof(uint64_t) * (size_t)(L.cgroups + 1));
    L.st_compact = take(sizeof(uint64_t) * (size_t)(L.fused_tiles + 1));
    L.st_emit = take(sizeof(uint64_t) * (size_t)(L.emit_tiles + 1));
    L.cidx = take(sizeof(uint32_t) * (size_t)un);
    L.sidx = take(sizeof(uint32_t) * (size_t)un);
    const size_t spec_slots =
        (hp.bin || hp.nospec) ? 0 : (size_t)L.ptiles * kSpecSlots;  // DGC selection only
    L.sval = take(sizeof(float) * spec_slots);
    L.su = take(sizeof(float) * spec_slots);
    L.tcount = take(sizeof(uint32_t) * (size_t)(L.ptiles + 1));
    L.tseg = take(sizeof(uint32_t) * (size_t)(L.ptiles + 1));
    L.eseg = take(sizeof(uint32_t) * 2 * (size_t)(L.emit_tiles + 1));
    L.clip_cnt = take(sizeof(uint32_t) * (size_t)nseg);
    L.dlist = take(sizeof(uint32_t) * (size_t)(L.ptiles + 1));
    L.binmax = take(sizeof(uint32_t) * (size_t)L.max_bins);
    L.total = o;
    return L;
}

uint64_t max_out_for(int64_t n, int32_t nseg, const HostParams& hp) {
    const uint64_t un = (uint64_t)n;
    if (hp.mode == DGC_SELECT_ADACOMP) return un;
    uint64_t ksum = count_ppb(un, hp.d_ppb) + (uint64_t)nseg;  // >= sum of per-segment ceils
    if (hp.d_ppb == 0) ksum = 0;
    uint64_t bound = ksum;
    if (hp.mode == DGC_SELECT_SAMPLED) {
        // no re-selection means |C| * 1e9 <= q * k, i.e. |S| <= floor(q * k / 1e9) per segment
        const unsigned __int128 b = (unsigned __int128)hp.q_ppb * ksum / kBillion + (uint64_t)nseg;
        bound = b > un ? un : (uint64_t)b;
    }
    return bound < un ? bound : un;
}

// Everything the kernels need, passed by value.
struct Args {
    const float* g;
    float* u;
    float* v;
    uint32_t n;
    int32_t nseg;
    const int64_t* seg_off;
    HostParams hp;
    uint32_t* out_idx;
    float* out_val;
    uint64_t out_cap;
    int64_t* out_count;
    dgc_seg_stats* stats;
    int32_t* status;
    Ctl* ctl;
    SampleCache* scache;
    SegInfo* segs;
    uint32_t* seg_start;
    uint32_t* samp_off;
    uint32_t* clip_off;
    uint32_t* cand_off;
    unsigned long long* clip_acc;  // per segment: the exact sum of squares (kSqWords words)
    uint32_t* skeys;
    uint32_t* spos;    // sample positions in ascending order (cached between calls)
    uint32_t* bcount;  // per-bucket counts, then cursors, while the cache is rebuilt
    uint32_t* histA;
    uint32_t* histB;
    uint64_t* st_collect;
    uint64_t* st_compact;
    uint64_t* st_emit;
    uint32_t* cidx;   // candidates, ascending index
    uint32_t* sidx;   // per-tile candidate slots of the streaming pass
    float* cval;      // candidate values v[cidx[f]] (in sidx's memory, once the slots are moved)
    float* sval;      // DGC pass: per tile with <= kSpecSlots candidates, their v values, by rank
    float* su;        // ... and their u values (kept with masking)
    uint32_t* tcount; // per-tile candidate counts, then (k_collect) each tile's first position
    uint32_t* tseg;   // streaming tile t starts in segment tseg[t]; tseg[ptiles] = nseg - 1
    uint32_t* eseg;   // emit tile t's candidates lie in segments [eseg[2t], eseg[2t + 1]]
    uint32_t* clip_cnt;  // clip tiles of each segment summed so far
    uint32_t* dlist;     // the streaming tiles with many candidates (k_collect_copy's work)
    uint32_t* binmax; // AdaComp: largest |v| key of every bin
    uint64_t max_samples, fused_tiles, emit_tiles, max_clip_tiles, ptiles, cgroups, nbuckets,
        max_bins;
    uint32_t spin_limit;
};

// ------------------------------------------------------------------------------- plan
// Block 0 builds the segment table; every block zeroes its share of the histograms and
// look-back words.
__global__ void __launch_bounds__(1024) k_plan(Args a) {
    __shared__ uint32_t s_scan[33];
    __shared__ uint32_t s_carry_samp, s_carry_clip, s_carry_bkt, s_carry_bin;
    __shared__ int s_bad;
    if (blockIdx.x == 0) {
        if (threadIdx.x == 0) {
            s_carry_samp = 0;
            s_carry_clip = 0;
            s_carry_bkt = 0;
            s_carry_bin = 0;
            s_bad = (a.seg_off[0] != 0 || a.seg_off[a.nseg] != (int64_t)a.n) ? 1 : 0;
            Ctl c{};
            *a.ctl = c;
            if (a.out_count) *a.out_count = 0;
        }
        __syncthreads();
        uint32_t active = 0;
        uint64_t tag = 0;  // what the sample positions depend on: seeds, ranges, counts
        for (int base = 0; base < a.nseg; base += 1024) {
            const int s = base + threadIdx.x;
            uint32_t ms = 0, clip_tiles = 0, buckets = 0, bins = 0;
            if (s < a.nseg) {
                const int64_t lo = a.seg_off[s], hi = a.seg_off[s + 1];
                if (hi < lo || lo < 0 || hi > (int64_t)a.n) atomicExch(&s_bad, 1);
                const uint32_t st = (uint32_t)min(max(lo, (int64_t)0), (int64_t)a.n);
                const uint32_t en = (uint32_t)min(max(hi, (int64_t)st), (int64_t)a.n);
                const uint32_t ns = en - st;
                SegInfo d{};
                d.start = st;
                d.end = en;
                d.k = a.hp.bin ? (ns + a.hp.bin - 1) / a.hp.bin  // AdaComp: bins
                               : (uint32_t)count_ppb(ns, a.hp.d_ppb);
                d.seed = mix64(a.hp.seed + kGolden * ((uint64_t)s + 1));
                d.scale = 1.0f;
                d.min_key = 0xFFFFFFFFu;
                d.thresh = kNoKey;
                if (d.k > 0 && a.hp.mode != DGC_SELECT_ADACOMP) {
                    if (a.hp.mode == DGC_SELECT_SAMPLED) {
                        d.ms = (uint32_t)count_ppb(ns, a.hp.r_ppb);
                        d.rank = (uint32_t)count_ppb(d.ms, a.hp.d_ppb);
                    } else if (ns >= kExactWholeBelow) {
                        const uint32_t m = (uint32_t)count_ppb(ns, a.hp.r_ppb);
                        const uint32_t ks = (uint32_t)count_ppb(m, a.hp.d_ppb);
                        const uint32_t margin = (uint32_t)ceilf(4.0f * sqrtf((float)ks)) + 16u;
                        if ((uint64_t)ks + margin < m) {
                            d.ms = m;
                            d.rank = ks + margin;
                        }
                    }
                    if (d.ms == 0) d.thresh = 0;  // exact mode, every entry a candidate
                    if (d.ms > 0) {
                        d.state = kActive;
                        d.need = d.rank;
                        ++active;
                    }
                }
                ms = d.ms;
                if (ms) buckets = (ns >> kBucketShift) + 1;
                if (a.hp.bin) bins = d.k;
                if (a.hp.clip_on) clip_tiles = (ns + kClipTile - 1) / kClipTile;
                a.segs[s] = d;
                a.seg_start[s] = st;
                tag ^= mix64(d.seed ^ mix64(((uint64_t)st << 32) | en) ^ mix64(ms + kGolden));
            }
            uint32_t tot;
            const uint32_t ex = block_excl_scan<1024>(ms, s_scan, &tot);
            if (s < a.nseg) a.samp_off[s] = s_carry_samp + ex;
            __syncthreads();
            if (threadIdx.x == 0) s_carry_samp += tot;
            const uint32_t exc = block_excl_scan<1024>(clip_tiles, s_scan, &tot);
            if (s < a.nseg) a.clip_off[s] = s_carry_clip + exc;
            __syncthreads();
            if (threadIdx.x == 0) s_carry_clip += tot;
            const uint32_t exb = block_excl_scan<1024>(buckets, s_scan, &tot);
            if (s < a.nseg) a.segs[s].bbase = s_carry_bkt + exb;
            __syncthreads();
            if (threadIdx.x == 0) s_carry_bkt += tot;
            const uint32_t exn = block_excl_scan<1024>(bins, s_scan, &tot);
            if (s < a.nseg) a.segs[s].binbase = s_carry_bin + exn;
            __syncthreads();
            if (threadIdx.x == 0) s_carry_bin += tot;
            __syncthreads();
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tag ^= __shfl_xor_sync(kFull, tag, o);
        if ((threadIdx.x & 31) == 0) atomicXor((unsigned long long*)&a.ctl->tag, tag);
        active = warp_sum(active);
        if ((threadIdx.x & 31) == 0 && active) atomicAdd(&a.ctl->active, active);
        __syncthreads();
        if (threadIdx.x == 0) {
            a.samp_off[a.nseg] = s_carry_samp;
            a.clip_off[a.nseg] = s_carry_clip;
            a.seg_start[a.nseg] = a.n;
            a.ctl->total_samples = s_carry_samp;
            a.ctl->total_clip_tiles = s_carry_clip;
            atomicXor((unsigned long long*)&a.ctl->tag,
                      mix64((uint64_t)a.n ^ mix64((uint64_t)a.nseg + kCacheMagic)));
            if (s_bad) {
                a.ctl->abort = 1;
                report(a.status, DGC_EINVAL);
            }
        }
    }
    // zero histograms and look-back words (grid-stride over all blocks)
    const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    const size_t nh = (size_t)a.nseg * kHistBins;
    for (size_t i = tid; i < nh; i += stride) {
        a.histA[i] = 0;
        a.histB[i] = 0;
    }
    for (size_t i = tid; i <= a.fused_tiles; i += stride) a.st_compact[i] = 0;
    for (size_t i = tid; i <= a.cgroups; i += stride) a.st_collect[i] = 0;
    for (size_t i = tid; i <= a.emit_tiles; i += stride) a.st_emit[i] = 0;
    for (size_t i = tid; i < a.nbuckets; i += stride) a.bcount[i] = 0;
    for (size_t i = tid; i < a.max_bins; i += stride) a.binmax[i] = 0;
    for (size_t i = tid; i < (size_t)a.nseg; i += stride) a.clip_cnt[i] = 0;
    if (a.hp.clip_on)
        for (size_t i = tid; i < (size_t)a.nseg * kSqWords; i += stride) a.clip_acc[i] = 0;
    // the segment of every streaming tile's first entry, searched in the caller's offsets (when
    // they are invalid, block 0 raises abort and no later kernel reads this)
    for (size_t t = tid; t <= a.ptiles; t += stride)
        a.tseg[t] = (t == a.ptiles) ? (uint32_t)(a.nseg - 1)
                                    : (uint32_t)upper_bound_minus1(a.seg_off, a.nseg,
                                                                   (int64_t)(t * kPTile));
}

// ----------------------------------------------------------------------------- clipping
// The sum of squares of a segment, exactly, rounded once to binary64 (ties to even). Entry
// x = m 2^(e'-150) (m the 24-bit significand, e' = max(biased exponent, 1)) has the exact
// square M 2^(2e'-300), M = m^2 < 2^48; the segment keeps X = sum M 2^(2e'-2) (2e'-2 <= 506, at
// most 2^32 entries: X < 2^586) and S = X 2^-298. X lives in kSqDigits 64-bit words, word i
// worth 2^(32 i), which take plain atomic adds that nobody waits for, in any order. A block
// keeps its share of a segment in the same form in shared memory: every shared add is below
// 2^33 (digits_add's middle piece holds two digits' worth), a tile makes at most 8 x 2 + 4096
// of them to one word (two per warp window, one per entry below its window), and a block sums
// at most ceil(2^20 / grid) + 1 tiles of a segment (under 1800 with the 608-block grid), so a
// shared word stays below 2^56. The block then adds 32-bit digits to the segment's global words
// (its carries propagated first), once per block and segment, so a global word stays below
// 2^42; the carries are propagated once more, by k_clip_round. A host model of these integer
// steps, with the bounds asserted, is in tests/test_clip_scheme_host.py.

// words[i..] += x 2^(32 i + sh) for x < 2^64, sh < 32: three 32-bit pieces
__device__ __forceinline__ void digits_add(unsigned long long* words, int i, int sh,
                                           unsigned long long x) {
    const unsigned long long lo = (x & 0xFFFFFFFFull) << sh;  // < 2^63
    const unsigned long long hi = (x >> 32) << sh;            // < 2^63
    const unsigned long long d0 = lo & 0xFFFFFFFFull;
    const unsigned long long d1 = (lo >> 32) + (hi & 0xFFFFFFFFull);
    const unsigned long long d2 = hi >> 32;
    if (d0) atomicAdd(words + i, d0);
    if (d1) atomicAdd(words + i + 1, d1);  // < 2^33: two digits' worth, still far from overflow
    if (d2) atomicAdd(words + i + 2, d2);
}

// X 2^-298 to the nearest binary64, ties to even, from X in 64-bit limbs: the top 64 bits of
// X, the bits below them folded into a sticky bit, then 53 of them kept. X < 2^586, so the
// result is a normal number.
__device__ double limbs_round(const unsigned long long* x) {
    int h = kSqLimbs - 1;
    while (h > 0 && x[h] == 0ull) --h;
    if (x[h] == 0ull) return 0.0;
    const int t = 64 * h + 63 - __clzll((long long)x[h]);  // the top set bit of X
    unsigned long long top;  // bits t .. t-63 of X (zeros below bit 0)
    bool sticky = false;
    if (t < 64) {
        top = x[0] << (63 - t);
    } else {
        const int pos = t - 63, j = pos >> 6, sh = pos & 63;
        top = sh ? ((x[j] >> sh) | (x[j + 1] << (64 - sh))) : x[j];
        sticky = sh && (x[j] & ((1ull << sh) - 1ull)) != 0ull;
        for (int i = 0; i < j; ++i) sticky = sticky || x[i] != 0ull;
    }
    unsigned long long mant = top >> 11;  // 53 bits, the leading one at bit 52
    const bool half = (top >> 10) & 1ull;
    sticky = sticky || (top & 0x3FFull) != 0ull;
    int te = t;
    if (half && (sticky || (mant & 1ull))) {
        ++mant;
        if (mant >> 53) {
            mant >>= 1;
            ++te;
        }
    }
    // mant 2^(te - 52 - 298): biased exponent te - 298 + 1023
    const unsigned long long bits =
        ((unsigned long long)(te + 725) << 52) | (mant & 0xFFFFFFFFFFFFFull);
    return __longlong_as_double((long long)bits);
}

// (w1:w0) += (p1:p0), 128 bits
__device__ __forceinline__ void add128(unsigned long long& w0, unsigned long long& w1,
                                       unsigned long long p0, unsigned long long p1) {
    asm("add.cc.u64 %0, %0, %2;\n\taddc.u64 %1, %1, %3;" : "+l"(w0), "+l"(w1) : "l"(p0), "l"(p1));
}

// m << (sh mod 32), truncated to 32 bits (a funnel shift in wrap mode)
__device__ __forceinline__ uint32_t shl_wrap(uint32_t m, uint32_t sh) {
    uint32_t r;
    asm("shf.l.wrap.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(0u), "r"(m), "r"(sh));
    return r;
}

// An entry with raw exponent e and significand m into a band: band 1 (e >= ea) adds
// (m 2^(e - ea))^2 to A1, anything else adds (m 2^((e - eb) mod 32) mod 2^32)^2 to A2, modulo
// 2^64. For an entry of band 2 that is its exact (m 2^(e - eb))^2; an entry below band 2 adds a
// term of no meaning, which the caller takes back out (A2 is exact modulo 2^64, and the true
// band sum is below 2^64).
__device__ __forceinline__ void band_add(uint32_t e, uint32_t m, uint32_t ea, uint32_t eb,
                                         unsigned long long& A1, unsigned long long& A2) {
    asm("{\n\t.reg .pred p;\n\t.reg .u32 b, d, mm;\n\t"
        "setp.ge.u32 p, %2, %4;\n\t"
        "selp.u32 b, %4, %5, p;\n\t"
        "sub.u32 d, %2, b;\n\t"
        "shf.l.wrap.b32 mm, 0, %3, d;\n\t"
        "@p mad.wide.u32 %0, mm, mm, %0;\n\t"
        "@!p mad.wide.u32 %1, mm, mm, %1;\n\t}"
        : "+l"(A1), "+l"(A2)
        : "r"(e), "r"(m), "r"(ea), "r"(eb));
}

// 16 bytes from global to this thread's own shared memory, asynchronously (cp.async); the
// thread reads them back itself after cp.async.wait_group, so no block barrier is involved
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

constexpr uint32_t kWinTiles = 16;  // tiles a warp window holds before it is flushed
constexpr int kClipStages = 2;      // tiles of copies in flight per block, plus the one summed
constexpr size_t kClipSmem = (size_t)kClipStages * 4 * kThreads * 16;

// 4096-entry tiles of one segment each. Block b takes a contiguous range of the tiles (so its
// segment changes only at segment boundaries), and its warps work without block barriers: warp w
// of a tile holds entries [512 w, 512 w + 512), 16 per thread. Each thread copies its 16 entries
// of the next tile into its own shared-memory slots (cp.async) while it sums the current one.
//
// A thread sums its 16 squares in two 64-bit bands below its own largest entry: an entry of band
// b with e' = eb + d (d <= 6) adds (m 2^d)^2 = M 4^d, a 32-bit shift of the significand
// (m 2^d < 2^30) and one 32 x 32 -> 64-bit multiply-add, so a band sum stays below 2^64.
// What lies more than 13 binades under the thread's largest entry (rare) goes to the block's
// digit words in shared memory at once. The band sums then go into the thread's 128-bit window,
// whose lowest bit is bit lo = max(2 E - 68, 0) of X, where E is the largest e' the warp has
// seen since it opened the window (each term below 2^118 there). A warp keeps its window over
// up to kWinTiles tiles of a segment and reopens it when a tile brings a larger e' or the
// segment ends: the threads' windows are then summed across the warp (below 2^128: at most
// 2 kWinTiles terms per thread, or 16 per tile below 2^114 for a thread holding inf or NaN) and
// lane 0 adds the sum to the block's digits (shared atomic adds, each below 2^33). Band sums
// whose bit lies below lo go to the digits directly. When the block moves to another segment,
// and at its end, one thread propagates the carries of the shared words into 32-bit digits and
// adds those to the segment's words in global memory (each below 2^32, at most one add per
// block and segment).
__global__ void __launch_bounds__(kThreads, 4) k_clip_tiles(Args a) {
    __shared__ unsigned long long s_dig[kSqDigits];  // the block's share of the current segment
    __shared__ uint32_t s_flags;                     // 2: +inf seen; 4: NaN seen
    // each thread's slots of kClipStages tiles: [stage][4][kThreads] 16-byte words
    extern __shared__ __align__(16) uint4 s_buf[];
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) s_flags = 0;
    if (threadIdx.x < kSqDigits) s_dig[threadIdx.x] = 0ull;
    if (a.ctl->abort) return;  // written only by earlier kernels: the same in every thread
    __syncthreads();
    const uint32_t total = a.ctl->total_clip_tiles;
    const uint32_t c0 = (uint32_t)((uint64_t)total * blockIdx.x / gridDim.x);
    const uint32_t c1 = (uint32_t)((uint64_t)total * (blockIdx.x + 1) / gridDim.x);
    if (c0 >= c1) return;
    int s = upper_bound_minus1(a.clip_off, a.nseg, c0);
    // the block's digits into segment s's words: carries first, then one add per digit
    auto flush = [&](int seg) {
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned long long* X = a.clip_acc + (size_t)seg * kSqWords;
            unsigned long long carry = 0ull;
            for (int j = 0; j < kSqDigits; ++j) {
                const unsigned long long t = s_dig[j] + carry;
                if (t & 0xFFFFFFFFull) atomicAdd(X + j, t & 0xFFFFFFFFull);
                carry = t >> 32;
                s_dig[j] = 0ull;
            }
            if (s_flags) atomicOr(X + kSqDigits, (unsigned long long)s_flags);
            s_flags = 0;
        }
        __syncthreads();
    };
    // the warp's window: E, its lowest bit lo, the tiles it holds (0: closed), this thread's part
    uint32_t E = 0, ntw = 0;
    int lo = 0;
    unsigned long long w0 = 0ull, w1 = 0ull;
    auto warp_flush = [&]() {  // warp-uniform: every lane has the same ntw
        if (ntw == 0) return;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const unsigned long long o0 = __shfl_down_sync(kFull, w0, off);
            const unsigned long long o1 = __shfl_down_sync(kFull, w1, off);
            add128(w0, w1, o0, o1);
        }
        if (lane == 0) {  // W 2^lo: W < 2^128 in five 32-bit pieces from word lo / 32
            const int i = lo >> 5, sh = lo & 31;
            digits_add(s_dig, i, sh, w0);
            digits_add(s_dig, i + 2, sh, w1);
        }
        w0 = w1 = 0ull;
        ntw = 0;
    };
    // v 2^bit into the window when bit >= lo, else into the block's digits (v 2^(bit - lo) is
    // below 2^118: a band sum, v < 2^64, has bit - lo <= 54, a single square, v < 2^48, <= 66)
    auto place = [&](unsigned long long v, int bit) {
        if (v == 0ull) return;
        const int r = bit - lo;
        if (r >= 0) {
            const unsigned long long p0 = (r < 64) ? (v << r) : 0ull;
            const unsigned long long p1 =
                (r == 0) ? 0ull : (r < 64) ? (v >> (64 - r)) : (v << (r - 64));
            add128(w0, w1, p0, p1);
        } else {
            digits_add(s_dig, bit >> 5, bit & 31, v);
        }
    };
    // A segment in registers: its tiles [t0, t1), its entries [beg, beg + rm). A thread's 16
    // entries of a tile start at offset off in the segment (below 2^32: a segment has fewer than
    // 2^32 entries); they come by cp.async when they are 16 whole entries on a 16-byte boundary,
    // else by plain loads. The copies run kClipStages - 1 tiles ahead of the sums, with their
    // own segment registers.
    auto seg_regs = [&](int seg, uint32_t& t0, uint32_t& t1, uint32_t& beg, uint32_t& rm) {
        t0 = a.clip_off[seg];
        t1 = a.clip_off[seg + 1];
        beg = a.segs[seg].start;
        rm = a.segs[seg].end - beg;
    };
    auto whole = [](uint32_t beg, uint32_t rm, uint32_t off) {
        return ((beg + off) & 3u) == 0 && rm >= 16u && off <= rm - 16u;
    };
    uint32_t sc0, sc1, sbeg, rem;  // the segment being summed
    seg_regs(s, sc0, sc1, sbeg, rem);
    uint32_t ic = c0, ic0 = sc0, ic1 = sc1, ibeg = sbeg, irem = rem;  // the next tile to copy
    int is = s, istage = 0;
    auto issue_next = [&]() {  // one commit group per tile, empty past the block's last tile
        if (ic < c1) {
            if (ic == ic1) {
                while (is + 1 < a.nseg && a.clip_off[is + 1] <= ic) ++is;
                seg_regs(is, ic0, ic1, ibeg, irem);
            }
            const uint32_t o = (ic - ic0) * kClipTile + 16u * threadIdx.x;
            if (whole(ibeg, irem, o)) {
                const uint4* src = reinterpret_cast<const uint4*>(a.g + ((uint64_t)ibeg + o));
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    cp_async16(&s_buf[(istage * 4 + j) * kThreads + threadIdx.x], src + j);
            }
        }
        cp_async_commit();
        ++ic;
        istage = (istage + 1 == kClipStages) ? 0 : istage + 1;
    };
#pragma unroll
    for (int k = 0; k < kClipStages - 1; ++k) issue_next();
    int stage = 0;
    for (uint32_t c = c0; c < c1; ++c) {
        if (c == sc1) {  // block-uniform: the next segment with tiles
            warp_flush();
            flush(s);
            while (s + 1 < a.nseg && a.clip_off[s + 1] <= c) ++s;
            seg_regs(s, sc0, sc1, sbeg, rem);
        }
        issue_next();  // tile c + kClipStages - 1
        cp_async_wait<kClipStages - 1>();  // tile c's copies have landed
        const uint32_t off = (c - sc0) * kClipTile + 16u * threadIdx.x;
        const bool fast = whole(sbeg, rem, off);
        // the tile's 16 entries sit in this thread's slots (entries past the segment's end as 0);
        // they are read from there twice: for the largest and smallest, then for the bands
        uint4* my = &s_buf[stage * 4 * kThreads + threadIdx.x];
        if (!fast) {
            uint32_t t[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t e = off + (uint32_t)i;  // (off + i cannot wrap: off < 2^32 - 15)
                t[i] = (e < rem) ? __float_as_uint(a.g[(uint64_t)sbeg + e]) : 0u;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                my[j * kThreads] = make_uint4(t[4 * j], t[4 * j + 1], t[4 * j + 2], t[4 * j + 3]);
        }
        // the largest and smallest |x| bits, each shifted left by one (the sign bit dropped)
        uint32_t amax = 0, amin = 0xFFFFFFFFu;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 x = my[j * kThreads];
            const uint32_t v[4] = {x.x << 1, x.y << 1, x.z << 1, x.w << 1};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                amax = max(amax, v[q]);
                amin = min(amin, v[q]);
            }
        }
        const bool nonfinite = amax >= 0xFF000000u;
        // the thread's largest e' (inf and NaN count as 254: the sum is then inf or NaN anyway,
        // and every bound below still holds)
        const uint32_t et = max(min(amax >> 24, 254u), 1u);
        const uint32_t em = __reduce_max_sync(kFull, et);
        if (ntw == kWinTiles || (ntw != 0 && em > E)) warp_flush();
        if (ntw == 0) {
            E = em;
            lo = max(2 * (int)em - 68, 0);
        }
        ++ntw;
        uint32_t fl = 0;
        // entry by entry from the slots: raw exponent e and significand m (with its hidden bit)
        auto each = [&](auto&& f) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 x = my[j * kThreads];
                const uint32_t v[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    f((v[q] << 1) >> 24, (v[q] & 0x7FFFFFu) | 0x800000u, v[q] & 0x7FFFFFFFu);
            }
        };
        if (!nonfinite) {
            // band 1: e' in [ea, ea + 6]; band 2: e' in [eb, ea - 1]; smaller entries go to the
            // shared digits one by one
            const uint32_t ea = max(et, 7u) - 6u;
            const uint32_t eb = max(ea, 8u) - 7u;
            // A band holds normal entries only (eb >= 1): there the significand is the fraction
            // with its hidden bit. Band membership is read off the raw exponent e, so zeros and
            // subnormals (e = 0) fall below the bands.
            unsigned long long A1 = 0ull, A2 = 0ull;
            each([&](uint32_t e, uint32_t m, uint32_t) { band_add(e, m, ea, eb, A1, A2); });
            // the smallest entry's exponent below eb: some entry, maybe a zero, lies below the
            // bands (rare for gradients without exact zeros). Each such entry takes its term
            // back out of A2 and adds its square to the shared digits.
            if ((amin >> 24) < eb) {
                each([&](uint32_t e, uint32_t mb, uint32_t ax) {
                    if (e < eb) {
                        const uint32_t w = shl_wrap(mb, e - eb);
                        A2 -= (unsigned long long)w * w;
                        if (ax != 0u) {
                            const uint32_t m = e ? mb : ax;
                            const int at = 2 * (int)max(e, 1u) - 2;
                            digits_add(s_dig, at >> 5, at & 31, (unsigned long long)m * m);
                        }
                    }
                });
            }
            place(A1, 2 * (int)ea - 2);
            place(A2, 2 * (int)eb - 2);
        } else {  // a thread holding inf or NaN: entry by entry
            each([&](uint32_t e, uint32_t, uint32_t ax) {
                if (e == 0xFFu) {
                    fl |= (ax & 0x7FFFFFu) ? 4u : 2u;
                    return;
                }
                const uint32_t m = e ? ((ax & 0x7FFFFFu) | 0x800000u) : ax;
                place((unsigned long long)m * m, 2 * (int)max(e, 1u) - 2);
            });
        }
        if (fl) atomicOr(&s_flags, fl);
        stage = (stage + 1 == kClipStages) ? 0 : stage + 1;
    }
    warp_flush();
    flush(s);
}

// One thread per segment, after every tile is summed: propagate the carries of the segment's
// words into 32-bit digits, read them as 64-bit limbs, round once, and set scale = c / sqrt(S)
// when sqrt(S) > c (correctly rounded binary64 sqrt and division, rounded once to binary32).
// A segment without entries keeps S = 0 and scale 1.
__global__ void __launch_bounds__(128) k_clip_round(Args a) {
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= a.nseg || a.ctl->abort) return;
    const unsigned long long* X = a.clip_acc + (size_t)s * kSqWords;
    unsigned long long limb[kSqLimbs];
    unsigned long long carry = 0ull;
#pragma unroll
    for (int j = 0; j < kSqLimbs; ++j) {
        const unsigned long long t0 = X[2 * j] + carry;
        const unsigned long long t1 = X[2 * j + 1] + (t0 >> 32);
        limb[j] = (t0 & 0xFFFFFFFFull) | (t1 << 32);
        carry = t1 >> 32;
    }
    double S = limbs_round(limb);
    const unsigned long long flags = X[kSqDigits];
    if (flags & 4ull) S = __longlong_as_double(0x7FF8000000000000ll);
    else if (flags & 2ull) S = __longlong_as_double(0x7FF0000000000000ll);
    const double norm = sqrt(S);
    const double cn = (double)a.hp.clip_norm;
    a.segs[s].scale = (norm > cn) ? (float)(cn / norm) : 1.0f;
    a.segs[s].sumsq = S;
}

// v <- fma(leak, v, u): with leak = 1 this is the plain sum v + u, rounded once
__device__ __forceinline__ void accumulate(float g, float& u, float& v, float m, float scale,
                                           float leak) {
    const float gp = (scale != 1.0f) ? __fmul_rn(g, scale) : g;
    u = __fmaf_rn(m, u, gp);
    v = __fmaf_rn(leak, v, u);
}

// ----------------------------------------------------------------------- histograms
// Per-block histogram of one segment in shared memory, flushed to the segment's global
// histogram when the block moves to another segment or ends.
struct BlockHist {
    uint32_t* s;       // kHistBins entries in shared memory
    int cur;           // segment currently held, -1 none
    __device__ void flush(uint32_t* ghist, int nbins) {
        __syncthreads();
        if (cur >= 0)
            for (int b = threadIdx.x; b < nbins; b += blockDim.x) {
                const uint32_t x = s[b];
                if (x) {
                    atomicAdd(&ghist[(size_t)cur * kHistBins + b], x);
                    s[b] = 0;
                }
            }
        __syncthreads();
    }
};

// ------------------------------------------------------------- sample-position cache
// The sample positions depend only on the seed and the segment layout, and gathering g, u, v in
// position order is much kinder to HBM than in draw order. So the workspace keeps the positions
// sorted by 1024-entry bucket (segment by segment, so each segment's samples stay together), with
// a tag of what they depend on and a checksum of the array. Every call re-checks both (one read
// of the array) and rebuilds the cache when either differs -- a workspace that was reused for
// something else, or a new seed or layout, costs one counting sort by bucket and a sort inside
// each bucket, so the cached array is the sample positions in ascending order, segment by
// segment. (The threshold only depends on the multiset of sampled keys in any case.)
__device__ __forceinline__ uint32_t sample_position(const SegInfo& d, uint64_t j) {
    const uint64_t x = mix64(d.seed + kGolden * (j + 1));
    return d.start + (uint32_t)__umul64hi(x, (uint64_t)(d.end - d.start));
}

__device__ __forceinline__ uint64_t cache_term(uint32_t pos, uint64_t i) {
    return mix64((uint64_t)pos ^ (i * kGolden));
}

__device__ __forceinline__ uint64_t block_sum64(uint64_t x, uint64_t* sm) {
    uint64_t total;
    block_excl_scan<kThreads>(x, sm, &total);
    return total;
}

__device__ bool grid_barrier(const Args& a, int* s_ok);

// One cooperative launch: the checksum of the cached positions (when the header matches this
// call's tag), a grid barrier, and -- only when the cache does not match -- the rebuild: bucket
// counts, their scan (one block), every position into its bucket, each bucket sorted, and the
// checksum of the new array, with grid barriers between the steps. Words written by other
// blocks in an earlier step are read past L1.
__global__ void __launch_bounds__(kThreads) k_cache(Args a) {
    __shared__ uint64_t s_scan64[33];
    __shared__ uint32_t s_scan[33];
    __shared__ int s_bar, s_go;
    if (ld_relaxed_u32((const uint32_t*)&a.ctl->abort)) return;  // the same word for every block
    const SampleCache c = *a.scache;
    const uint64_t tag = a.ctl->tag;
    const bool tag_ok = c.magic == kCacheMagic && c.tag == tag;
    const uint32_t total = a.ctl->total_samples;
    const uint64_t tid = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    const uint64_t stride = (uint64_t)gridDim.x * kThreads;
    if (tag_ok) {
        uint64_t part = 0;
        // 16-byte loads of 4 positions (the array is 256-byte aligned), 4 of them in flight
        constexpr int kB = 4;
        const uint64_t total4 = total / 4;
        const uint4* sp4 = reinterpret_cast<const uint4*>(a.spos);
        for (uint64_t q0 = tid; q0 < total4; q0 += kB * stride) {
            uint4 p[kB];
#pragma unroll
            for (int r = 0; r < kB; ++r)
                p[r] = (q0 + r * stride < total4) ? sp4[q0 + r * stride] : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int r = 0; r < kB; ++r) {
                const uint64_t i = 4 * (q0 + r * stride);
                if (q0 + r * stride < total4)
                    part += cache_term(p[r].x, i) + cache_term(p[r].y, i + 1) +
                            cache_term(p[r].z, i + 2) + cache_term(p[r].w, i + 3);
            }
        }
        for (uint64_t i = 4 * total4 + tid; i < total; i += stride) part += cache_term(a.spos[i], i);
        const uint64_t sum = block_sum64(part, s_scan64);
        if (threadIdx.x == 0 && sum) atomicAdd((unsigned long long*)&a.ctl->csum, sum);
    }
    if (!grid_barrier(a, &s_bar)) return;
    if (threadIdx.x == 0) s_go = !(tag_ok && c.checksum == ld_relaxed(&a.ctl->csum));
    __syncthreads();
    if (!s_go) return;  // the cache matches: the same decision in every block
    // bucket counts
    for (uint64_t jg = tid; jg < total; jg += stride) {
        const int s = upper_bound_minus1(a.samp_off, a.nseg, (uint32_t)jg);
        const SegInfo& d = a.segs[s];
        const uint32_t pos = sample_position(d, jg - a.samp_off[s]);
        atomicAdd(&a.bcount[d.bbase + ((pos - d.start) >> kBucketShift)], 1u);
    }
    if (!grid_barrier(a, &s_bar)) return;
    // counts -> first slot of each bucket (block 0)
    if (blockIdx.x == 0) {
        const uint64_t nb = a.nbuckets;
        const uint64_t per = (nb + kThreads - 1) / kThreads;
        const uint64_t lo = umin64(nb, threadIdx.x * per), hi = umin64(nb, lo + per);
        uint32_t mine = 0;
        for (uint64_t b = lo; b < hi; ++b) mine += __ldcg(a.bcount + b);
        uint32_t sum;
        uint32_t run = block_excl_scan<kThreads>(mine, s_scan, &sum);
        for (uint64_t b = lo; b < hi; ++b) {
            const uint32_t n_b = __ldcg(a.bcount + b);
            a.bcount[b] = run;
            run += n_b;
        }
    }
    if (!grid_barrier(a, &s_bar)) return;
    // every position into its bucket; bcount[b] ends as the end of bucket b
    for (uint64_t jg = tid; jg < total; jg += stride) {
        const int s = upper_bound_minus1(a.samp_off, a.nseg, (uint32_t)jg);
        const SegInfo& d = a.segs[s];
        const uint32_t pos = sample_position(d, jg - a.samp_off[s]);
        const uint32_t slot = atomicAdd(&a.bcount[d.bbase + ((pos - d.start) >> kBucketShift)], 1u);
        a.spos[slot] = pos;
    }
    if (!grid_barrier(a, &s_bar)) return;
    // each bucket's positions in ascending order (about ten per bucket), so that the gather
    // walks every array upward
    for (uint64_t b = tid; b < a.nbuckets; b += stride) {
        const uint32_t lo = b ? __ldcg(a.bcount + b - 1) : 0u, hi = __ldcg(a.bcount + b);
        for (uint32_t i = lo + 1; i < hi; ++i) {  // insertion sort
            const uint32_t x = __ldcg(a.spos + i);
            uint32_t j = i;
            while (j > lo) {
                const uint32_t y = __ldcg(a.spos + j - 1);
                if (y <= x) break;
                a.spos[j] = y;
                --j;
            }
            a.spos[j] = x;
        }
    }
    if (!grid_barrier(a, &s_bar)) return;
    // checksum of the new array; block 0 writes the header once every block has added its part
    uint64_t part = 0;
    for (uint64_t i = tid; i < total; i += stride) part += cache_term(__ldcg(a.spos + i), i);
    const uint64_t sum = block_sum64(part, s_scan64);
    if (threadIdx.x == 0 && sum) atomicAdd((unsigned long long*)&a.ctl->newsum, sum);
    if (!grid_barrier(a, &s_bar)) return;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        SampleCache h;
        h.magic = kCacheMagic;
        h.tag = tag;
        h.checksum = ld_relaxed(&a.ctl->newsum);
        h.pad = 0;
        *a.scache = h;
    }
}

// --------------------------------------------------------------------------- sampling
// Sample draw j of segment s sits at start + floor(mix(seed_s + (j+1)g) * n_s / 2^64). The
// post-accumulate value there is recomputed from the pre-step g, u, v with the same
// operations the streaming pass uses, so it is bit-identical to what that pass will store.
//
// A scattered 4-byte load costs a whole DRAM burst, so this gather is bound by the bursts in
// flight: every thread issues its kSamplePerThread x 3 gathers before it uses any of them, and
// the grid holds one block per kThreads x kSamplePerThread samples, so that many blocks stay
// resident. (Persistent blocks walking rounds of 8 samples per thread, 24 gathers in flight,
// kept fewer warps resident and measured slower.) A block inside one segment counts into a
// shared histogram, one atomic per distinct bin per warp (lanes with equal bins found by
// __match_any_sync), and flushes it to the segment's global histogram at its end.
constexpr int kSamplePerThread = 4;

__global__ void __launch_bounds__(kThreads) k_sample(Args a) {
    __shared__ uint32_t s_hist[kHistBins];
    __shared__ int s_seg0, s_seg1, s_skip;
    if (threadIdx.x == 0) s_skip = a.ctl->abort;
    __syncthreads();
    if (s_skip) return;
    const uint32_t total = a.ctl->total_samples;
    const uint64_t chunk0 = (uint64_t)blockIdx.x * kThreads * kSamplePerThread;
    if (chunk0 >= total) return;
    for (int b = threadIdx.x; b < kHistBins; b += kThreads) s_hist[b] = 0;
    const uint64_t chunk_end = umin64(total, chunk0 + kThreads * kSamplePerThread);
    if (threadIdx.x == 0) {
        s_seg0 = upper_bound_minus1(a.samp_off, a.nseg, (uint32_t)chunk0);
        s_seg1 = upper_bound_minus1(a.samp_off, a.nseg, (uint32_t)(chunk_end - 1));
    }
    __syncthreads();
    const bool uniform = (s_seg0 == s_seg1);
    const int lane = threadIdx.x & 31;
    float gv[kSamplePerThread], uv[kSamplePerThread], vv[kSamplePerThread];
    int sg[kSamplePerThread];
#pragma unroll
    for (int r = 0; r < kSamplePerThread; ++r) {
        const uint64_t jg = chunk0 + r * kThreads + threadIdx.x;
        sg[r] = -1;
        if (jg < chunk_end) {
            // a chunk that crosses segments searches only its own segment range
            const int s = uniform ? s_seg0
                                  : s_seg0 + upper_bound_minus1(a.samp_off + s_seg0,
                                                                s_seg1 - s_seg0 + 1, (uint32_t)jg);
            const uint32_t pos = a.spos[jg];  // the sample positions in ascending order
            gv[r] = __ldg(a.g + pos);
            uv[r] = a.u[pos];
            vv[r] = a.v[pos];
            sg[r] = s;
        }
    }
#pragma unroll
    for (int r = 0; r < kSamplePerThread; ++r) {
        const uint64_t jg = chunk0 + r * kThreads + threadIdx.x;
        const bool valid = sg[r] >= 0;
        uint32_t bin = 0;
        if (valid) {
            float uu = uv[r], vn = vv[r];
            accumulate(gv[r], uu, vn, a.hp.momentum, a.segs[sg[r]].scale, a.hp.leak);
            const uint32_t key = key_of(vn);
            a.skeys[jg] = key;
            bin = key >> 20;
        }
        if (uniform) {  // block-uniform branch: every lane of the warp is here
            const unsigned m = __ballot_sync(kFull, valid);
            if (valid) {
                const unsigned peers = __match_any_sync(m, bin);
                if (lane == __ffs(peers) - 1) atomicAdd(&s_hist[bin], (uint32_t)__popc(peers));
            }
        } else if (valid) {
            atomicAdd(&a.histA[(size_t)sg[r] * kHistBins + bin], 1u);
        }
    }
    if (uniform) {
        BlockHist h{s_hist, s_seg0};
        h.flush(a.histA, kHistBins);
    }
}

// ----------------------------------------------------------------- radix select: hist
// Items are the sample keys (kind 0: X = key << 32) or the candidates (kind 1:
// X = key << 32 | ~index). Level L counts, per active segment, the items whose bits above the
// level match the prefix found so far, by the level's digit.
template <int kKind>
__device__ __forceinline__ uint64_t item_x(const Args& a, uint32_t i) {
    if (kKind == 0) return (uint64_t)a.skeys[i] << 32;
    return ((uint64_t)key_of(a.cval[i]) << 32) | (uint64_t)(~a.cidx[i]);
}

// Runs inside the cooperative select, where other blocks change the segment words between
// levels: those are read past L1 (ld.global.cg).
// With `compact` (the sample select's second level) every item that matches its segment's
// prefix is also appended to a compact list -- its key in the slot array's memory, its segment
// in the candidate list's, both unused until the streaming pass -- so that the third level
// counts only those (hist_compact).
constexpr uint32_t kCompBuf = 1024;  // kept keys a block gathers before one global append
__device__ __forceinline__ void compact_push(const Args& a, uint32_t* s_ck, uint32_t* s_cs,
                                             uint32_t* s_cn, uint32_t key, uint32_t seg) {
    const uint32_t q = atomicAdd(s_cn, 1u);
    if (q < kCompBuf) {
        s_ck[q] = key;
        s_cs[q] = seg;
    } else {  // the block's buffer is full: straight to the list
        const uint32_t pos = atomicAdd(&a.ctl->ncomp, 1u);
        if (pos < a.n) {
            a.sidx[pos] = key;
            a.cidx[pos] = seg;
        }
    }
}

template <int kKind>
__device__ void hist_level(const Args& a, int level, uint32_t* s_hist, bool compact) {
    __shared__ uint32_t s_ck[kCompBuf], s_cs[kCompBuf];
    __shared__ uint32_t s_cn, s_cbase;
    if (threadIdx.x == 0) s_cn = 0;
    const uint32_t* off = kKind == 0 ? a.samp_off : a.cand_off;
    const uint32_t total = off[a.nseg];
    uint32_t* ghist = (level & 1) ? a.histB : a.histA;
    const int shift = c_shift[level], bits = c_bits[level];
    const int nbins = 1 << bits;
    const uint32_t mask = (uint32_t)nbins - 1;
    for (int b = threadIdx.x; b < kHistBins; b += kThreads) s_hist[b] = 0;
    __syncthreads();
    BlockHist h{s_hist, -1};
    constexpr int kPer = 16;
    const uint32_t chunk = kThreads * kPer;
    // the segment words do not change during a level: read them again only when the chunk's
    // segment changes (every thread holds the same copy)
    int seen = -1;
    bool seen_active = false;
    uint64_t seen_prefix = 0;
    for (uint64_t c0 = (uint64_t)blockIdx.x * chunk; c0 < total; c0 += (uint64_t)gridDim.x * chunk) {
        const uint32_t c1 = (uint32_t)umin64(total, c0 + chunk);
        const int s0 = upper_bound_minus1(off, a.nseg, (uint32_t)c0);
        const int s1 = upper_bound_minus1(off, a.nseg, c1 - 1);
        if (s0 == s1) {
            if (s0 != seen) {
                seen = s0;
                seen_active = __ldcg(&a.segs[s0].state) == kActive;
                seen_prefix = __ldcg(&a.segs[s0].prefix);
            }
            if (!seen_active) continue;
            if (h.cur != s0) {
                h.flush(ghist, nbins);
                h.cur = s0;
            }
            const uint64_t prefix = seen_prefix;
            uint64_t xs[kPer];
#pragma unroll
            for (int r = 0; r < kPer; ++r) {  // all loads first, then the counting
                const uint32_t i = (uint32_t)c0 + r * kThreads + threadIdx.x;
                xs[r] = (i < c1) ? item_x<kKind>(a, i) : ~0ull;
            }
#pragma unroll
            for (int r = 0; r < kPer; ++r) {
                const uint32_t i = (uint32_t)c0 + r * kThreads + threadIdx.x;
                if (i < c1 && (xs[r] >> (shift + bits)) == prefix) {
                    atomicAdd(&s_hist[(xs[r] >> shift) & mask], 1u);
                    if (compact) compact_push(a, s_ck, s_cs, &s_cn, (uint32_t)(xs[r] >> 32), s0);
                }
            }
        } else {
            for (uint32_t i = (uint32_t)c0 + threadIdx.x; i < c1; i += kThreads) {
                const int s = s0 + upper_bound_minus1(off + s0, s1 - s0 + 1, i);
                const SegInfo& d = a.segs[s];
                if (__ldcg(&d.state) != kActive) continue;
                const uint64_t x = item_x<kKind>(a, i);
                if ((x >> (shift + bits)) == __ldcg(&d.prefix)) {
                    atomicAdd(&ghist[(size_t)s * kHistBins + ((x >> shift) & mask)], 1u);
                    if (compact) compact_push(a, s_ck, s_cs, &s_cn, (uint32_t)(x >> 32), (uint32_t)s);
                }
            }
        }
    }
    h.flush(ghist, nbins);  // ends with a barrier: the block's kept keys are all in s_ck
    if (compact) {  // one global append for the block's kept keys
        const uint32_t m = min(s_cn, kCompBuf);
        if (threadIdx.x == 0) s_cbase = m ? atomicAdd(&a.ctl->ncomp, m) : 0u;
        __syncthreads();
        for (uint32_t q = threadIdx.x; q < m; q += kThreads) {
            const uint32_t pos = s_cbase + q;
            if (pos < a.n) {
                a.sidx[pos] = s_ck[q];
                a.cidx[pos] = s_cs[q];
            }
        }
    }
}

// The sample select's third level over the compact list the second level left (key, segment),
// written by other blocks before the grid barrier: read past L1.
__device__ void hist_compact(const Args& a, int level) {
    const uint32_t nc = (uint32_t)umin64(ld_relaxed_u32(&a.ctl->ncomp), a.n);
    uint32_t* ghist = (level & 1) ? a.histB : a.histA;
    const int shift = c_shift[level], bits = c_bits[level];
    const uint32_t mask = (1u << bits) - 1u;
    for (uint32_t i = blockIdx.x * kThreads + threadIdx.x; i < nc; i += gridDim.x * kThreads) {
        const uint32_t s = __ldcg(a.cidx + i);
        const uint64_t x = (uint64_t)__ldcg(a.sidx + i) << 32;
        const SegInfo& d = a.segs[s];
        if (__ldcg(&d.state) != kActive) continue;
        if ((x >> (shift + bits)) == __ldcg(&d.prefix))
            atomicAdd(&ghist[(size_t)s * kHistBins + ((x >> shift) & mask)], 1u);
    }
}

// ----------------------------------------------------------------- radix select: find
// Walk the bins of `hist` from the top until `need` items are covered (block-wide, kBlock
// threads; thread t owns the positions [t*per, t*per + per) counted from the top bin down).
// After the call's barrier r->found says whether the walk ended inside the histogram, r->bin
// is that bin, r->above the items in higher bins and r->cnt the bin's own count. The bins read
// are set to zero afterwards (visible after the caller's next barrier).
struct FindRes {
    uint32_t bin, above, cnt;
    int found;
};

template <int kBlock, bool kCG = false>
__device__ void find_from_top(uint32_t* hist, int nbins, uint32_t need, uint32_t* s_scan,
                              FindRes* r) {
    constexpr int kMaxPer = kHistBins / kBlock;
    const int per = nbins / kBlock;
    uint32_t h[kMaxPer];
    uint32_t local = 0;
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i) {
        h[i] = 0;
        if (i < per) {
            const uint32_t* p = hist + (nbins - 1 - (threadIdx.x * per + i));
            h[i] = kCG ? __ldcg(p) : *p;
            local += h[i];
        }
    }
    if (threadIdx.x == 0) r->found = 0;
    uint32_t tot;
    const uint32_t ex = block_excl_scan<kBlock>(local, s_scan, &tot);
    if (ex < need && need <= ex + local) {
        uint32_t cum = ex;
#pragma unroll
        for (int i = 0; i < kMaxPer; ++i) {
            if (i < per && cum < need && need <= cum + h[i]) {
                r->bin = (uint32_t)(nbins - 1 - (threadIdx.x * per + i));
                r->above = cum;
                r->cnt = h[i];
                r->found = 1;
            }
            cum += (i < per) ? h[i] : 0;
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i)
        if (i < per) hist[nbins - 1 - (threadIdx.x * per + i)] = 0;
}

// One level's outcome: the bin extends the prefix. True when the selection is complete: for
// the sample select the prefix after three levels is the threshold key t; for the candidate
// select, once the bin holds exactly the items still needed (or at the last level), everything
// at or above prefix << shift is selected.
template <int kKind>
__device__ __forceinline__ bool select_step(int level, int bits, const FindRes& r,
                                            uint64_t& prefix, uint32_t& need) {
    prefix = (prefix << bits) | r.bin;
    const uint32_t need2 = need - r.above;
    need = need2;
    return kKind == 0 ? level == 2 : (r.cnt == need2 || level == 5);
}

// The end of a segment's select: the threshold key (kind 0) or sel_x (kind 1).
template <int kKind>
__device__ __forceinline__ void select_done(const Args& a, SegInfo& d, bool found, int level,
                                            uint64_t prefix) {
    if (!found) {  // fewer items than needed: cannot happen for a consistent table
        report(a.status, DGC_EINVAL);
        d.sel_x = 0;
    } else if (kKind == 0) {
        d.thresh = (uint32_t)prefix;
    } else {
        d.sel_x = prefix << c_shift[level];
    }
    d.state = kIdle;
    atomicSub(&a.ctl->active, 1u);
}

// Grid-wide barrier of a cooperative launch (every block resident). Thread 0 of each block
// arrives on a counter; the last arrival resets it and bumps the generation the others poll.
// The poll is bounded: past spin_limit the block reports DGC_ETIMEOUT, raises abort and
// returns false (so does every block that then sees abort).
__device__ bool grid_barrier(const Args& a, int* s_ok) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t g = ld_relaxed_u32(&a.ctl->bar_gen);
        __threadfence();
        int ok = 1;
        if (atomicAdd(&a.ctl->bar_count, 1u) == gridDim.x - 1) {
            a.ctl->bar_count = 0;
            __threadfence();
            atomicExch(&a.ctl->bar_gen, g + 1);
        } else {
            uint32_t spins = 0;
            while (ld_relaxed_u32(&a.ctl->bar_gen) == g) {
                if (++spins > a.spin_limit) {
                    report(a.status, DGC_ETIMEOUT);
                    atomicExch(&a.ctl->abort, 1);
                    ok = 0;
                    break;
                }
                __nanosleep(64);
            }
        }
        __threadfence();
        *s_ok = ok && !ld_relaxed_u32((const uint32_t*)&a.ctl->abort);
    }
    __syncthreads();
    return *s_ok != 0;
}

// The global-memory radix select for the segments the on-chip select left active, every level
// in one cooperative launch: a level counts (all blocks, grid-stride over the items; the sample
// select's third level only over the keys its second level kept), then
// after a grid barrier blocks take the active segments and walk their histograms from the top,
// then a grid barrier. The sample select's first level was counted by the sampling
// kernel. The kernel ends as soon as no segment is active, at once when none was to begin
// with. Segment words and histograms change between levels, so they are read past L1.
template <int kKind>
__global__ void __launch_bounds__(kThreads) k_select_global(Args a) {
    __shared__ uint32_t s_hist[kHistBins];
    __shared__ uint32_t s_scan[33];
    __shared__ FindRes s_r;
    __shared__ int s_go, s_bar;
    constexpr int kLevels = kKind == 0 ? 3 : 6;
    if (threadIdx.x == 0)
        s_go = !ld_relaxed_u32((const uint32_t*)&a.ctl->abort) &&
               ld_relaxed_u32(&a.ctl->active) != 0;
    __syncthreads();
    if (!s_go) return;  // the same words for every block: no block reaches a barrier alone
    for (int level = 0; level < kLevels; ++level) {
        const int bits = c_bits[level];
        if (kKind == 1 || level > 0) {
            if (kKind == 0 && level == 2)
                hist_compact(a, level);
            else
                hist_level<kKind>(a, level, s_hist, kKind == 0 && level == 1);
            if (!grid_barrier(a, &s_bar)) return;
        }
        uint32_t* hbase = (level & 1) ? a.histB : a.histA;
        for (int s = blockIdx.x; s < a.nseg; s += gridDim.x) {
            SegInfo& d = a.segs[s];
            if (__ldcg(&d.state) != kActive) continue;  // only this block changes it, below
            const uint32_t need0 = __ldcg(&d.need);
            find_from_top<kThreads, true>(hbase + (size_t)s * kHistBins, 1 << bits, need0,
                                          s_scan, &s_r);
            if (threadIdx.x == 0) {
                uint64_t prefix = __ldcg(&d.prefix);
                uint32_t need = need0;
                if (!s_r.found || select_step<kKind>(level, bits, s_r, prefix, need)) {
                    select_done<kKind>(a, d, s_r.found, level, prefix);
                } else {
                    d.prefix = prefix;
                    d.need = need;
                }
            }
        }
        if (!grid_barrier(a, &s_bar)) return;
        if (threadIdx.x == 0) s_go = ld_relaxed_u32(&a.ctl->active) != 0;
        __syncthreads();
        if (!s_go) return;
    }
}

// ------------------------------------------------------ radix select: whole segment on chip
// One block per active segment whose items fit in shared memory: every level runs on chip, and
// each level keeps only the items that still match the prefix (each warp compacts its own share
// in place). Segments with more items stay active for the global-memory levels
// (k_select_global). The segment's contiguous items (sample keys, or candidate indices and
// values) arrive by bulk copy; candidate values become keys and are counted for the first
// level on chip. For the sample select
// the first level's counts come from the sampling kernel's histogram, cleared here as the global
// walk would. Two blocks fit on an SM, so up to 2 x 152 segments run in one wave.
constexpr int kSmallThreads = 512;
constexpr size_t kSmallBytes = 100u * 1024u;
template <int kKind>
__global__ void __launch_bounds__(kSmallThreads, 2) k_select_small(Args a) {
    constexpr uint32_t kArrays = kKind == 0 ? 1 : 2;  // sample keys | candidate indices, keys
    // the copy starts at the 16-byte boundary at or before the first item: 3 words of slack
    constexpr uint32_t kCap = (uint32_t)(kSmallBytes / (4 * kArrays)) - 4;
    constexpr int kW = kSmallThreads / 32;
    constexpr int kLevels = kKind == 0 ? 3 : 6;
    extern __shared__ __align__(16) unsigned char s_dyn[];
    __shared__ uint32_t s_hist[kHistBins];
    __shared__ uint32_t s_scan[33];
    __shared__ FindRes s_r;
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ int s_fail;
    const int s = blockIdx.x;
    SegInfo& d = a.segs[s];
    if (a.ctl->abort || d.state != kActive) return;  // every thread reads the same words
    const uint32_t* off = kKind == 0 ? a.samp_off : a.cand_off;
    const uint32_t i0 = off[s], C = off[s + 1] - i0;
    if (C > kCap) return;
    uint32_t* sraw = reinterpret_cast<uint32_t*>(s_dyn);
    uint32_t* s_a = sraw + (i0 & 3u);  // item i: key (kind 0) or candidate index (kind 1)
    uint32_t* s_k = sraw + kCap + 4 + (i0 & 3u);  // kind 1: the value, then the key, of item i
    if (threadIdx.x == 0) {
        s_fail = 0;
        mbar_init(&s_bar, 1);
        mbar_init_fence();
        // whole 16-byte units from the boundary at or before item 0; the workspace regions are
        // padded to 256 bytes, so the last unit stays inside the array's region
        const uint32_t bytes = (((i0 & 3u) + C + 3u) & ~3u) * 4u;
        mbar_arrive_expect_tx(&s_bar, kKind == 0 ? bytes : 2u * bytes);
        if (bytes) bulk_g2s(sraw, (kKind == 0 ? a.skeys : a.cidx) + (i0 & ~3u), bytes, &s_bar);
        if (kKind == 1 && bytes)
            bulk_g2s(sraw + kCap + 4, a.cval + (i0 & ~3u), bytes, &s_bar);
    }
    constexpr int kBinsPer = kHistBins / kSmallThreads;
    if (kKind == 0) {  // all of the thread's bins in flight at once, then cleared
        uint32_t* gh = a.histA + (size_t)s * kHistBins;
        uint32_t hv[kBinsPer];
#pragma unroll
        for (int r = 0; r < kBinsPer; ++r) hv[r] = gh[threadIdx.x + r * kSmallThreads];
#pragma unroll
        for (int r = 0; r < kBinsPer; ++r) {
            s_hist[threadIdx.x + r * kSmallThreads] = hv[r];
            gh[threadIdx.x + r * kSmallThreads] = 0;
        }
    } else {
        for (int b = threadIdx.x; b < kHistBins; b += kSmallThreads) s_hist[b] = 0;
    }
    __syncthreads();  // the mbarrier is initialised before anyone polls it
    {
        uint32_t spins = 0;
        while (!mbar_try_wait(&s_bar, 0)) {
            if (++spins > kMbarSpinLimit) {
                s_fail = 1;
                break;
            }
        }
    }
    __syncthreads();
    if (s_fail) {  // the copy never landed: report, give it one more bounded wait, leave
        if (threadIdx.x == 0) {
            report(a.status, DGC_ETIMEOUT);
            atomicExch(&a.ctl->abort, 1);
        }
        for (uint32_t k = 0; k < kMbarSpinLimit && !mbar_try_wait(&s_bar, 0); ++k) {
        }
        return;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t R = (C + kW - 1) / kW;
    const uint32_t wb = min(C, (uint32_t)warp * R), we = min(C, wb + R);
    uint32_t wn = we - wb;  // items this warp still holds, at the front of its share
    if (kKind == 1) {
        // values to keys, counted for the first level; candidates crowd into a few first-level
        // bins, so lanes with the same bin add once
        for (uint32_t j = wb; j < we + 31u; j += 32) {
            const uint32_t i = j + lane;
            const bool in = i < we && j < we;
            const uint32_t key = in ? (s_k[i] & 0x7FFFFFFFu) : 0u;
            const uint32_t bin = in ? key >> 20 : 0xFFFFFFFFu;  // X >> 52
            const unsigned peers = __match_any_sync(kFull, bin);
            if (in) {
                s_k[i] = key;
                if (lane == __ffs(peers) - 1) atomicAdd(&s_hist[bin], (uint32_t)__popc(peers));
            }
        }
        __syncthreads();
    }
    uint64_t prefix = 0;
    uint32_t need = d.need;
    bool done = false, found = true;
    int level = 0;
    for (; level < kLevels; ++level) {
        const int shift = c_shift[level], bits = c_bits[level];
        const uint32_t mask = (1u << bits) - 1u;
        if (level > 0) {
            uint32_t keep = 0;
            for (uint32_t j = 0; j < wn; j += 32) {
                const bool in = j + lane < wn;
                const uint32_t ia = in ? s_a[wb + j + lane] : 0u;
                const uint32_t ik = (kKind == 1 && in) ? s_k[wb + j + lane] : 0u;
                const uint64_t x = kKind == 0 ? ((uint64_t)ia << 32)
                                              : (((uint64_t)ik << 32) | (uint64_t)(~ia));
                const bool match = in && (x >> (shift + bits)) == prefix;
                const unsigned mm = __ballot_sync(kFull, match);
                if (match) {
                    atomicAdd(&s_hist[(uint32_t)(x >> shift) & mask], 1u);
                    // write position <= every position read in this round: in place is safe
                    const uint32_t w = wb + keep + __popc(mm & ((1u << lane) - 1u));
                    s_a[w] = ia;
                    if (kKind == 1) s_k[w] = ik;
                }
                keep += __popc(mm);
            }
            wn = keep;
            __syncthreads();
        }
        find_from_top<kSmallThreads>(s_hist, 1 << bits, need, s_scan, &s_r);
        __syncthreads();
        if (!s_r.found) {
            found = false;
            break;
        }
        if (select_step<kKind>(level, bits, s_r, prefix, need)) {
            done = true;
            break;
        }
    }
    if (threadIdx.x == 0) select_done<kKind>(a, d, found && done, min(level, kLevels - 1), prefix);
}

// ------------------------------------------------------------- exact-mode re-compaction
// Runs only when, in exact mode, a segment's sampled lower bound admitted fewer than k
// candidates: it rebuilds the whole index-ordered candidate list from v (already updated),
// with threshold 0 for those segments. One tile per block, offsets by decoupled look-back.
__global__ void __launch_bounds__(kThreads, 2) k_recompact(Args a) {
    __shared__ uint32_t s_bitmap[kTile / 32];
    __shared__ uint32_t s_wordpre[kTile / 32];
    __shared__ uint32_t s_scan[33];
    __shared__ uint32_t s_tile;
    __shared__ uint64_t s_base;
    __shared__ int s_uniform, s_skip;
    __shared__ uint32_t s_thresh;
    const uint64_t n = a.n;
    // one thread reads the flags and takes the tile, so the whole block agrees
    if (threadIdx.x == 0) {
        s_skip = !a.ctl->any_failed || ld_relaxed_u32((const uint32_t*)&a.ctl->abort);
        if (!s_skip) s_tile = atomicAdd(&a.ctl->ticket_compact, 1u);
    }
    for (int w = threadIdx.x; w < kTile / 32; w += kThreads) s_bitmap[w] = 0;
    __syncthreads();
    if (s_skip) return;
    const uint32_t tile = s_tile;
    const uint64_t base = (uint64_t)tile * kTile;
    const uint64_t tile_end = umin64(n, base + kTile);
    if (threadIdx.x == 0) {
        const SegInfo& d = a.segs[upper_bound_minus1(a.seg_start, a.nseg, (uint32_t)base)];
        s_uniform = (d.end >= tile_end) ? 1 : 0;
        s_thresh = d.failed ? 0u : d.thresh;
    }
    __syncthreads();
    uint32_t flags = 0;  // bit r*4+e: entry e of row r is a candidate
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        const uint64_t e0 = base + 4u * (r * kThreads + threadIdx.x);
        uint32_t f4 = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (e0 + e >= n) continue;
            uint32_t t = s_thresh;
            if (!s_uniform) {
                const SegInfo& d =
                    a.segs[upper_bound_minus1(a.seg_start, a.nseg, (uint32_t)(e0 + e))];
                t = d.failed ? 0u : d.thresh;
            }
            if (key_of(a.v[e0 + e]) >= t) f4 |= 1u << e;
        }
        if (f4) {
            const uint32_t off = (uint32_t)(e0 - base);
            atomicOr(&s_bitmap[off >> 5], f4 << (off & 31));
        }
        flags |= f4 << (4 * r);
    }
    __syncthreads();
    static_assert(kTile / 32 == kThreads, "one bitmap word per thread");
    const uint32_t cnt = __popc(s_bitmap[threadIdx.x]);
    uint32_t tile_total;
    s_wordpre[threadIdx.x] = block_excl_scan<kThreads>(cnt, s_scan, &tile_total);
    if (threadIdx.x < 32) {
        const uint64_t excl = lookback_exclusive(a.st_compact, tile, tile_total, a.spin_limit,
                                                 a.status, &a.ctl->abort);
        if (threadIdx.x == 0) s_base = excl;
    }
    __syncthreads();
    const uint64_t gbase = s_base;
#pragma unroll
    for (int q = 0; q < kRows * 4; ++q) {
        if (!(flags & (1u << q))) continue;
        const uint32_t off = 4u * ((q >> 2) * kThreads + threadIdx.x) + (q & 3);
        const uint32_t w = off >> 5;
        const uint64_t pos = gbase + s_wordpre[w] + __popc(s_bitmap[w] & ((1u << (off & 31)) - 1u));
        if (pos < n) a.cidx[pos] = (uint32_t)(base + off);
    }
    if (tile == a.fused_tiles - 1 && threadIdx.x == 0)
        a.ctl->total_cand = (uint32_t)umin64(gbase + tile_total, n);
}

// ------------------------------------------------- streaming pass, bulk-copy pipeline
// The pass every entry goes through: u = fma(m, u, g*scale); v += u; candidates are the
// entries with key(v) >= the segment's threshold. Persistent blocks (2 or 3 per SM) take
// kPTile-entry tiles from an atomic ticket and keep 4 or 3 tiles of g, u and v in flight as bulk copies
// (TMA, cp.async.bulk) into shared memory, so HBM streams without pause. Updated u and v go back
// with coalesced 16-byte stores. A tile's candidates are compacted, in index order, into the
// tile's own slot range sidx[base, base + count) and its count into tcount[tile]: no block
// ever waits on another, and k_collect turns the counts into global offsets afterwards.
// In a tile that crosses a segment boundary, entry i lies in one of the segments
// [s0, s0 + ns) (from the tile table), found by a short search.
__device__ __forceinline__ const SegInfo& tile_segment(const Args& a, int s0, int ns, uint32_t i) {
    return a.segs[s0 + upper_bound_minus1(a.seg_start + s0, ns, i)];
}

template <bool kKeepU>
__device__ __forceinline__ void stream_compute(const Args& a, const float* sg, uint64_t base,
                                               uint32_t len, bool uniform, int s0, int ns,
                                               float scale0, uint32_t thresh0,
                                               float4 (&uu)[kPRows], float4 (&vv)[kPRows],
                                               uint32_t& flags) {
    const int tid = threadIdx.x;
    const uint32_t bulk = len & ~3u;
    flags = 0;
#pragma unroll
    for (int r = 0; r < kPRows; ++r) {
        const uint32_t off = 4u * (r * kThreads + tid);
        float4 g4, u4, v4;
        if (off + 4 <= bulk) {
            g4 = reinterpret_cast<const float4*>(sg)[r * kThreads + tid];
            u4 = reinterpret_cast<const float4*>(sg + kPTile)[r * kThreads + tid];
            v4 = reinterpret_cast<const float4*>(sg + 2 * kPTile)[r * kThreads + tid];
        } else {  // the last, ragged tile: at most 3 entries past the bulk copy
            float tg[4], tu[4], tv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool in = off + e < len;
                tg[e] = in ? a.g[base + off + e] : 0.f;
                tu[e] = in ? a.u[base + off + e] : 0.f;
                tv[e] = in ? a.v[base + off + e] : 0.f;
            }
            g4 = make_float4(tg[0], tg[1], tg[2], tg[3]);
            u4 = make_float4(tu[0], tu[1], tu[2], tu[3]);
            v4 = make_float4(tv[0], tv[1], tv[2], tv[3]);
        }
        float* gp = reinterpret_cast<float*>(&g4);
        float* up = reinterpret_cast<float*>(&u4);
        float* vp = reinterpret_cast<float*>(&v4);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (off + e >= len) continue;
            float scale = scale0;
            uint32_t t = thresh0;
            if (!uniform) {
                const SegInfo& d = tile_segment(a, s0, ns, (uint32_t)(base + off + e));
                scale = d.scale;
                t = d.thresh;
            }
            accumulate(gp[e], up[e], vp[e], a.hp.momentum, scale, a.hp.leak);
            if (key_of(vp[e]) >= t) flags |= 1u << (4 * r + e);
        }
        if (kKeepU) uu[r] = u4;
        vv[r] = v4;
    }
}

// Row r of a thread's updated u and v back to memory: one 16-byte store each, entry by entry
// in the ragged last tile.
__device__ __forceinline__ void store_uv(const Args& a, uint64_t base, uint32_t len, int r,
                                         int tid, const float4& u4, const float4& v4) {
    const uint32_t off = 4u * (r * kThreads + tid);
    if (off + 4 <= len) {
        *reinterpret_cast<float4*>(a.u + base + off) = u4;
        *reinterpret_cast<float4*>(a.v + base + off) = v4;
    } else {
        const float* u2 = reinterpret_cast<const float*>(&u4);
        const float* v2 = reinterpret_cast<const float*>(&v4);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (off + e < len) {
                a.u[base + off + e] = u2[e];
                a.v[base + off + e] = v2[e];
            }
    }
}

// kSel 0: candidates are the entries at or above the segment's threshold key (DGC). kSel 1
// (AdaComp): candidates are the entries at the largest key of their bin within the tile; the
// tile also raises each bin's global maximum, and the emit step keeps the candidates that
// reach it. kSel 2 (a shared index set given by the caller): the pass only accumulates.
template <int kSel>
__global__ void __launch_bounds__(kThreads, stream_blocks_per_sm<kSel>()) k_stream_tma(Args a) {
    constexpr int kPStages = stream_stages<kSel>();
    extern __shared__ __align__(128) float s_stage[];  // [kPStages][3][kPTile]
    __shared__ __align__(8) uint64_t s_bar[kPStages];
    __shared__ uint32_t s_tile[kPStages];
    __shared__ int s_uniform[kPStages];
    __shared__ int s_seg0[kPStages], s_nseg[kPStages];  // the tile's segments [s0, s0 + ns)
    __shared__ float s_scale[kPStages];
    __shared__ uint32_t s_thresh[kPStages];
    __shared__ uint32_t s_binA[kPStages];  // AdaComp: global index of the tile's first bin
    __shared__ uint32_t s_rem[kPStages];   // AdaComp: offset of the tile start in bin s_binA
    __shared__ uint32_t s_rc[2][kPRows * kWarps];  // candidates per (row, warp), by parity
    __shared__ int s_skip;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t n = a.n;
    const uint32_t ntiles = (uint32_t)((n + kPTile - 1) / kPTile);

    // thread 0 owns the pipeline: it takes a ticket, notes the tile's segments, and starts the
    // tile's three bulk copies; the mbarrier phase publishes all of it to the block. Tickets are
    // taken two issues ahead and their tile-table entries read one issue ahead, so neither the
    // atomic's round trip nor the table read (a miss while HBM streams) waits in line with the
    // copies. Tickets rise within a block, so the block stops at its first tile past the end
    // having handled every tile it took before; the tickets it still holds are past the end.
    uint32_t t_next = 0, t_next2 = 0;  // the next two tickets
    uint32_t s0_next = 0, s1_next = 0;  // tile-table entries of t_next (read when t_next < ntiles)
    auto issue = [&](int st) {
        const uint32_t t = t_next;
        const int s0 = (int)s0_next, s1 = (int)s1_next;
        t_next = t_next2;
        if (t_next < ntiles) {
            s0_next = a.tseg[t_next];
            s1_next = a.tseg[t_next + 1];
        }
        t_next2 = atomicAdd(&a.ctl->ticket_fused, 1u);
        s_tile[st] = t;
        if (t < ntiles) {
            const uint64_t base = (uint64_t)t * kPTile;
            const uint32_t len = (uint32_t)umin64(kPTile, n - base);
            const SegInfo& d = a.segs[s0];
            s_seg0[st] = s0;
            s_nseg[st] = s1 - s0 + 1;
            s_uniform[st] = (d.end >= base + len) ? 1 : 0;
            s_scale[st] = d.scale;
            s_thresh[st] = d.thresh;
            if (kSel == 1) {
                const uint32_t binA = d.binbase + ((uint32_t)base - d.start) / a.hp.bin;
                s_binA[st] = binA;
                s_rem[st] = ((uint32_t)base - d.start) - (binA - d.binbase) * a.hp.bin;
            }
            const uint32_t bytes = (len & ~3u) * 4u;  // whole 16-byte units; the rest by hand
            mbar_arrive_expect_tx(&s_bar[st], 3u * bytes);
            if (bytes) {
                float* dst = s_stage + (size_t)st * kPStageFloats;
                bulk_g2s(dst, a.g + base, bytes, &s_bar[st]);
                bulk_g2s(dst + kPTile, a.u + base, bytes, &s_bar[st]);
                bulk_g2s(dst + 2 * kPTile, a.v + base, bytes, &s_bar[st]);
            }
        } else {
            mbar_arrive_expect_tx(&s_bar[st], 0u);  // an empty phase marks the end
        }
    };

    if (tid == 0) {
        s_skip = ld_relaxed_u32((const uint32_t*)&a.ctl->abort);
        if (!s_skip) {
            for (int st = 0; st < kPStages; ++st) mbar_init(&s_bar[st], 1);
            mbar_init_fence();
            t_next = atomicAdd(&a.ctl->ticket_fused, 1u);
            t_next2 = atomicAdd(&a.ctl->ticket_fused, 1u);
            if (t_next < ntiles) {
                s0_next = a.tseg[t_next];
                s1_next = a.tseg[t_next + 1];
            }
            for (int st = 0; st < kPStages; ++st) issue(st);
        }
    }
    __syncthreads();
    if (s_skip) return;

    for (uint32_t it = 0;; ++it) {
        const int st = (int)(it % kPStages);
        const uint32_t parity = (it / kPStages) & 1u;
        uint32_t spins = 0;
        while (!mbar_try_wait(&s_bar[st], parity)) {
            if (++spins > kMbarSpinLimit) {  // a bulk copy that never lands: report, give the
                if (tid == 0) {              // copy one more bounded wait, then leave
                    report(a.status, DGC_ETIMEOUT);
                    atomicExch(&a.ctl->abort, 1);
                }
                for (uint32_t k = 0; k < kMbarSpinLimit && !mbar_try_wait(&s_bar[st], parity); ++k) {
                }
                return;
            }
        }
        const uint32_t tile = s_tile[st];
        if (tile >= ntiles) break;  // every later stage holds an empty phase too
        const uint64_t base = (uint64_t)tile * kPTile;
        const uint32_t len = (uint32_t)(umin64(n, base + kPTile) - base);
        float4 uu[kPRows], vv[kPRows];
        uint32_t flags;
        stream_compute<true>(a, s_stage + (size_t)st * kPStageFloats, base, len, s_uniform[st],
                             s_seg0[st], s_nseg[st], s_scale[st], s_thresh[st], uu, vv, flags);
        if constexpr (kSel == 2) flags = 0;  // the shared set is given: no candidates
        if constexpr (kSel == 1) {
            // AdaComp without a block barrier: each warp row (128 consecutive entries) finds the
            // largest key of every run of one bin inside it, raises the bin's global maximum with
            // it, and makes the entries that reach their run's maximum candidates. A bin's
            // global maximum is the largest of its runs' maxima, so every entry the emit step
            // keeps (key == the bin's global maximum) is a candidate. Entries past len hold
            // v = 0 (key 0): they raise nothing and are never candidates.
            const uint32_t binA = s_binA[st], L = a.hp.bin;
            uint32_t* gmax = a.binmax + binA;  // global maxima, indexed by local bin
            flags = 0;
            if (s_uniform[st] && L >= 4u) {
                // one segment: tile entry o lies in local bin (rem + o) / L, rem being the tile
                // start's offset within bin binA. A lane's 4 entries span at most two bins, and
                // bins rise with o, so a warp row holds contiguous runs of equal bins.
                const uint32_t rem = s_rem[st];
#pragma unroll
                for (int r = 0; r < kPRows; ++r) {
                    const uint32_t o0 = 4u * (r * kThreads + tid);
                    uint32_t q, d0;  // the lane's first local bin; entries before the next one
                    if (L >= (uint32_t)kPTile) {
                        q = (o0 >= L - rem) ? 1u : 0u;
                        d0 = q ? L - (o0 - (L - rem)) : L - rem - o0;
                    } else {  // (x + 0.5) * fl(1/L) rounds down to x / L here (x < 2 kPTile)
                        const uint32_t x = rem + o0;
                        q = __float2uint_rd(__fmul_rn(__fadd_rn((float)x, 0.5f), a.hp.bin_inv));
                        d0 = L - (x - q * L);
                    }
                    const float* vr = reinterpret_cast<const float*>(&vv[r]);
                    const uint32_t kk[4] = {key_of(vr[0]), key_of(vr[1]), key_of(vr[2]),
                                            key_of(vr[3])};
                    const bool split = d0 < 4u;  // the first bin ends inside this lane (rare)
                    uint32_t mlo, mhi = 0;
                    if (!split) {
                        mlo = max(max(kk[0], kk[1]), max(kk[2], kk[3]));
                    } else {
                        mlo = kk[0];  // d0 >= 1: entry 0 is always in the first bin
                        mhi = d0 <= 1u ? kk[1] : 0u;
                        mlo = d0 > 1u ? max(mlo, kk[1]) : mlo;
                        mhi = d0 <= 2u ? max(mhi, kk[2]) : mhi;
                        mlo = d0 > 2u ? max(mlo, kk[2]) : mlo;
                        mhi = max(mhi, kk[3]);  // d0 <= 3
                    }
                    const uint32_t b = q + (split ? 1u : 0u);  // the lane's last bin
                    uint32_t run;  // the maximum of the lane's last bin over the row
                    if (L >= 128u) {  // at most two bins in the row's 128 entries
                        const uint32_t b0 = __shfl_sync(kFull, b, 0), b1 = __shfl_sync(kFull, b, 31);
                        const uint32_t mx = split ? mhi : mlo;
                        if (b0 == b1) {  // the whole row in one bin (the common case)
                            run = __reduce_max_sync(kFull, mx);
                            if (lane == 0 && run) atomicMax(gmax + b0, run);
                        } else {
                            const uint32_t m0 = __reduce_max_sync(kFull, b == b0 ? mx : 0u);
                            const uint32_t m1 = __reduce_max_sync(kFull, b == b1 ? mx : 0u);
                            if (lane == 0 && m0) atomicMax(gmax + b0, m0);
                            if (lane == 31 && m1) atomicMax(gmax + b1, m1);
                            run = (b == b0) ? m0 : m1;
                        }
                    } else {  // segmented max by shuffles, suffix then prefix over each run
                        run = split ? mhi : mlo;
#pragma unroll
                        for (int dl = 1; dl < 32; dl <<= 1) {
                            const uint32_t om = __shfl_down_sync(kFull, run, dl);
                            const uint32_t ob = __shfl_down_sync(kFull, b, dl);
                            if (lane + dl < 32 && ob == b && om > run) run = om;
                        }
                        const uint32_t pb = __shfl_up_sync(kFull, b, 1);
                        if (run && (lane == 0 || pb != b)) atomicMax(gmax + b, run);
#pragma unroll
                        for (int dl = 1; dl < 32; dl <<= 1) {
                            const uint32_t om = __shfl_up_sync(kFull, run, dl);
                            const uint32_t ob = __shfl_up_sync(kFull, b, dl);
                            if (lane >= dl && ob == b && om > run) run = om;
                        }
                    }
                    // the first bin of a split lane: its run ends here, and the lane before
                    // holds the row's maximum of it when that lane's last bin is the same
                    const uint32_t prun = __shfl_up_sync(kFull, run, 1);
                    const uint32_t pbin = __shfl_up_sync(kFull, b, 1);
                    if (split) {
                        const uint32_t rq = (lane > 0 && pbin == q) ? max(prun, mlo) : mlo;
                        if (lane == 0 || pbin != q) {  // this lane holds the whole run
                            if (mlo) atomicMax(gmax + q, mlo);
                        } else if (rq > prun) {  // the lane before did not see this part
                            atomicMax(gmax + q, rq);
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const uint32_t m = ((uint32_t)e < d0) ? rq : run;
                            if (kk[e] && kk[e] == m) flags |= 1u << (4 * r + e);
                        }
                    } else if (run && mlo == run) {  // this lane reaches its run's maximum
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (kk[e] == run) flags |= 1u << (4 * r + e);
                    }
                }
            } else {  // a segment boundary inside the tile, or bins under 4 entries: every
                      // non-zero entry is a candidate and raises its bin's maximum itself
#pragma unroll
                for (int r = 0; r < kPRows; ++r)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t off = 4u * (r * kThreads + tid) + e;
                        const uint32_t key = key_of(reinterpret_cast<const float*>(&vv[r])[e]);
                        if (off < len && key) {
                            const uint32_t i = (uint32_t)(base + off);
                            const SegInfo& d = tile_segment(a, s_seg0[st], s_nseg[st], i);
                            atomicMax(a.binmax + d.binbase + (i - d.start) / L, key);
                            flags |= 1u << (4 * r + e);
                        }
                    }
            }
        }
        // candidate words: the 8 lanes of a lane-group cover 32 consecutive entries of a row
        uint32_t word[kPRows];
#pragma unroll
        for (int r = 0; r < kPRows; ++r) {
            uint32_t x = ((flags >> (4 * r)) & 0xFu) << (4 * (lane & 7));
            x |= __shfl_xor_sync(kFull, x, 1);
            x |= __shfl_xor_sync(kFull, x, 2);
            x |= __shfl_xor_sync(kFull, x, 4);
            word[r] = x;
            const uint32_t pc = __popc(x);
            const uint32_t rc = __shfl_sync(kFull, pc, 0) + __shfl_sync(kFull, pc, 8) +
                                __shfl_sync(kFull, pc, 16) + __shfl_sync(kFull, pc, 24);
            if (lane == 0) s_rc[it & 1][r * kWarps + warp] = rc;
            // rows without a candidate of this thread store now; the DGC pass stores the others
            // once the tile's count has decided whether they are sent speculatively
            if (kSel != 0 || ((flags >> (4 * r)) & 0xFu) == 0u)
                store_uv(a, base, len, r, tid, uu[r], vv[r]);
        }
        __syncthreads();  // the stage's data is in registers, the per-(row, warp) counts in place
        if (tid == 0) {
            fence_proxy_async_smem();
            issue(st);  // the next tile for this stage starts loading now
        }
        // every warp scans the kPRows x kWarps counts itself (row-major = index order)
        const uint32_t cv = (lane < kPRows * kWarps) ? s_rc[it & 1][lane] : 0u;
        const uint32_t cinc = warp_incl_scan(cv);
        const uint32_t tile_total = __shfl_sync(kFull, cinc, 31);
        // DGC pass: a tile with few candidates (nearly every tile at high sparsity) sends them
        // speculatively -- v (and u, with masking) is stored as 0 there, the values go to the
        // tile's kSpecSlots value slots -- so the emit step need not scatter the zeros; it puts
        // back the few candidates the selection then leaves out
        const bool spec = (kSel == 0) && !a.hp.nospec && tile_total <= kSpecSlots;
#pragma unroll
        for (int r = 0; r < kPRows; ++r) {  // every lane joins the shuffles, candidates or not
            const uint32_t f4 = (flags >> (4 * r)) & 0xFu;
            // entries before this lane's: earlier (row, warp) chunks, earlier lane-groups of this
            // chunk, earlier lanes of this lane-group
            const int ci = r * kWarps + warp;
            uint32_t before = __shfl_sync(kFull, cinc, ci) - __shfl_sync(kFull, cv, ci);
            const uint32_t p0 = __popc(__shfl_sync(kFull, word[r], 0));
            const uint32_t p1 = __popc(__shfl_sync(kFull, word[r], 8));
            const uint32_t p2 = __popc(__shfl_sync(kFull, word[r], 16));
            const int grp = lane >> 3;
            before += (grp > 0 ? p0 : 0) + (grp > 1 ? p1 : 0) + (grp > 2 ? p2 : 0);
            const uint32_t sh = 4u * (lane & 7);
            if (f4) {
                float* up = reinterpret_cast<float*>(&uu[r]);
                float* vp = reinterpret_cast<float*>(&vv[r]);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (f4 & (1u << e)) {
                        const uint32_t rank = before + __popc(word[r] & ((1u << (sh + e)) - 1u));
                        a.sidx[base + rank] = (uint32_t)(base + 4u * (r * kThreads + tid) + e);
                        if (spec) {
                            const size_t slot = (size_t)tile * kSpecSlots + rank;
                            a.sval[slot] = vp[e];
                            vp[e] = 0.0f;
                            if (a.hp.mask) {
                                a.su[slot] = up[e];
                                up[e] = 0.0f;
                            }
                        }
                    }
            }
            if (kSel == 0 && f4) store_uv(a, base, len, r, tid, uu[r], vv[r]);
        }
        if (tid == 0) a.tcount[tile] = tile_total;
    }
}

// ------------------------------------------------------------------------- collect
// Turns the streaming pass's per-tile slots into one index-ordered candidate list. Block b owns
// kCGroup consecutive tiles: it scans their counts and gets the group's global offset from a
// decoupled look-back over groups; each tile's count is replaced by its first list position. A
// tile's few candidates are copied to cidx by its own thread; tiles with more are listed for
// k_collect_copy.
constexpr int kCGroup = kThreads;  // tiles per collect block
constexpr uint32_t kCollectDirect = 16;  // a tile with at most this many candidates: copied in place
constexpr uint32_t kCollectWarp = 256;   // up to this many: one warp; more: one block

__global__ void __launch_bounds__(kThreads) k_collect(Args a) {
    __shared__ uint32_t s_scan[33];
    __shared__ uint64_t s_lb64[33];
    __shared__ uint32_t s_lb32[2];
    __shared__ uint32_t s_group;
    __shared__ int s_skip;
    const int tid = threadIdx.x;
    const uint32_t ntiles = (uint32_t)a.ptiles;
    const uint32_t ngroups = (ntiles + kCGroup - 1) / kCGroup;
    if (tid == 0) {
        s_skip = ld_relaxed_u32((const uint32_t*)&a.ctl->abort);
        if (!s_skip) s_group = atomicAdd(&a.ctl->ticket_collect, 1u);
    }
    __syncthreads();
    if (s_skip) return;
    const uint32_t grp = s_group;
    if (grp >= ngroups) return;
    const uint32_t t = grp * kCGroup + tid;
    const uint32_t c = (t < ntiles) ? a.tcount[t] : 0u;
    uint32_t total;
    const uint32_t ex = block_excl_scan<kThreads>(c, s_scan, &total);
    // the group's offset: a look-back walked by the whole block (kThreads groups per round trip)
    const uint64_t gbase = block_lookback<kThreads>(a.st_collect, grp, total, a.spin_limit,
                                                    a.status, &a.ctl->abort, s_lb32, s_lb64);
    // the tile's count becomes its first position in the list. A tile with few candidates (the
    // common case) has its slots copied by its own thread; the others are listed for
    // k_collect_copy, which spreads each over a whole block.
    if (t < ntiles) {
        const uint32_t p = (uint32_t)umin64(gbase + ex, a.n);
        a.tcount[t] = p;
        if (c <= kCollectDirect) {
            uint32_t x[kCollectDirect];
#pragma unroll
            for (uint32_t j = 0; j < kCollectDirect; ++j)
                if (j < c) x[j] = a.sidx[(uint64_t)t * kPTile + j];
#pragma unroll
            for (uint32_t j = 0; j < kCollectDirect; ++j)
                if (j < c && (uint64_t)p + j < a.n) a.cidx[p + j] = x[j];
        } else if (c <= kCollectWarp) {
            a.dlist[atomicAdd(&a.ctl->ndense, 1u)] = t;
        } else {
            a.dlist[ntiles - atomicAdd(&a.ctl->nlarge, 1u)] = t;
        }
    }
    if (grp == ngroups - 1 && tid == 0)
        a.ctl->total_cand = (uint32_t)umin64(gbase + total, a.n);
}

// The listed tiles' slots. A tile with more than kCollectWarp candidates (a run of small
// all-candidate segments) is copied by a whole block. The others -- with AdaComp's bins nearly
// every tile -- by a warp each: a warp reads the positions of 32 list entries at once (entries
// spread over the warps) and then copies those tiles one after another.
__global__ void __launch_bounds__(kThreads) k_collect_copy(Args a) {
    if (ld_relaxed_u32((const uint32_t*)&a.ctl->abort)) return;
    const uint32_t total = a.ctl->total_cand;
    const uint32_t nt = (uint32_t)a.ptiles;
    const uint32_t nd = a.ctl->ndense, nl = a.ctl->nlarge;
    for (uint32_t j = blockIdx.x; j < nl; j += gridDim.x) {
        const uint32_t t = a.dlist[nt - j];
        const uint32_t p = a.tcount[t];
        const uint32_t e = (t + 1 < nt) ? a.tcount[t + 1] : total;
        for (uint32_t q = threadIdx.x; p + q < e; q += kThreads)
            a.cidx[p + q] = a.sidx[(uint64_t)t * kPTile + q];
    }
    const int lane = threadIdx.x & 31;
    const uint64_t warps = (uint64_t)gridDim.x * kWarps;
    for (uint64_t jb = (uint64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); jb < nd;
         jb += 32 * warps) {
        const uint64_t j = jb + lane * warps;
        uint32_t t = 0, p = 0, e = 0;
        if (j < nd) {
            t = a.dlist[j];
            p = a.tcount[t];
            e = (t + 1 < nt) ? a.tcount[t + 1] : total;
        }
        const int m = (int)umin64(32, (nd - jb + warps - 1) / warps);  // entries jb + k warps < nd
        for (int k = 0; k < m; ++k) {
            const uint32_t tk = __shfl_sync(kFull, t, k), pk = __shfl_sync(kFull, p, k);
            const uint32_t ek = __shfl_sync(kFull, e, k);
            for (uint32_t q = lane; pk + q < ek; q += 32)
                a.cidx[pk + q] = a.sidx[(uint64_t)tk * kPTile + q];
        }
    }
}

// The value slot of candidate f (list position; index idx) when its streaming tile sent it
// speculatively (kept its v and u there and stored zeros), else -1: AdaComp, tiles with more than
// kSpecSlots candidates, and every tile once the exact mode's re-compaction has undone the zeros.
// After k_collect, tcount[t] is tile t's first list position, and its candidates follow in rank
// order, so f - tcount[t] is the rank the streaming pass gave f.
__device__ __forceinline__ int64_t spec_slot(const Args& a, uint64_t f, uint32_t idx,
                                             uint32_t total, bool unspec) {
    if (a.hp.bin || a.hp.nospec || unspec) return -1;
    const uint32_t t = idx / kPTile;
    const uint32_t first = a.tcount[t];
    const uint32_t next = (t + 1 < (uint32_t)a.ptiles) ? a.tcount[t + 1] : total;
    if (next - first > kSpecSlots) return -1;
    return (int64_t)t * kSpecSlots + (int64_t)(f - first);
}

// Every candidate's value, gathered once by the whole grid into cval (the slot array's memory,
// free once k_collect / k_collect_copy have moved the slots): from its tile's value slots when
// it was sent speculatively (v holds 0 there), else from v. The selects and the emit step then
// read values in list order, instead of each block gathering its segment's share from one SM.
__global__ void __launch_bounds__(kThreads) k_cval(Args a) {
    if (ld_relaxed_u32((const uint32_t*)&a.ctl->abort)) return;
    const uint64_t total = a.ctl->total_cand;
    const bool unspec = ld_relaxed_u32(&a.ctl->unspec) != 0;
    const uint64_t stride = (uint64_t)gridDim.x * kThreads;
    constexpr int kB = 4;  // gathers in flight per thread
    for (uint64_t f0 = (uint64_t)blockIdx.x * kThreads + threadIdx.x; f0 < total; f0 += kB * stride) {
        uint32_t idx[kB];
#pragma unroll
        for (int r = 0; r < kB; ++r) idx[r] = (f0 + r * stride < total) ? a.cidx[f0 + r * stride] : 0u;
        float x[kB];
#pragma unroll
        for (int r = 0; r < kB; ++r) {
            const uint64_t f = f0 + r * stride;
            x[r] = 0.0f;
            if (f < total) {
                const int64_t slot = spec_slot(a, f, idx[r], (uint32_t)total, unspec);
                x[r] = slot >= 0 ? a.sval[slot] : a.v[idx[r]];
            }
        }
#pragma unroll
        for (int r = 0; r < kB; ++r)
            if (f0 + r * stride < total) a.cval[f0 + r * stride] = x[r];
    }
}

// Exact mode, only when a segment's sampled bound admitted fewer than k candidates: before the
// re-compaction reads v again, every speculatively sent candidate gets its v and u back, and no
// later kernel of the call treats any tile as speculative.
__global__ void __launch_bounds__(kThreads) k_unspec(Args a) {
    if (ld_relaxed_u32((const uint32_t*)&a.ctl->abort) || !ld_relaxed_u32(&a.ctl->any_failed))
        return;
    const uint32_t total = a.ctl->total_cand;
    for (uint64_t f = (uint64_t)blockIdx.x * kThreads + threadIdx.x; f < total;
         f += (uint64_t)gridDim.x * kThreads) {
        const uint32_t idx = a.cidx[f];
        const int64_t slot = spec_slot(a, f, idx, total, false);
        if (slot >= 0) {
            a.v[idx] = a.sval[slot];
            if (a.hp.mask) a.u[idx] = a.su[slot];
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) a.ctl->unspec = 1;
}

// ------------------------------------------------------------------- candidate ranges
// One block: per-segment candidate ranges by binary search of the ascending candidate
// indices, then who selects among them. pass 1 only runs after an exact-mode re-compaction.
// In pass 0 the list is still laid out by streaming tile (k_collect left each tile's first
// position in tcount), so the first candidate at or past x lies in x's tile's own range.
constexpr int kCandoffStage = 4096;  // segment ranges staged in shared memory below this many
__global__ void __launch_bounds__(1024) k_candoff(Args a, int pass) {
    __shared__ uint32_t s_coff[kCandoffStage];
    __shared__ uint32_t s_active;
    __shared__ int s_skip;
    if (threadIdx.x == 0) s_skip = a.ctl->abort || (pass == 1 && !a.ctl->any_failed);
    __syncthreads();
    if (s_skip) return;
    if (threadIdx.x == 0) {
        a.ctl->active = 0;
        s_active = 0;
    }
    const uint32_t total = a.ctl->total_cand;
    const uint32_t ntiles = (uint32_t)a.ptiles;
    for (int s = threadIdx.x; s <= a.nseg; s += blockDim.x) {
        const uint32_t x = a.seg_start[s];
        uint32_t lo = 0, hi = total;  // first candidate index >= x
        const uint32_t t = x / kPTile;
        if (pass == 0 && t < ntiles) {
            lo = a.tcount[t];
            hi = (t + 1 < ntiles) ? a.tcount[t + 1] : total;
            // the tile's candidates ascend through [t kPTile, (t+1) kPTile): probe the position
            // the tile's density predicts, and its left neighbour (exact when every entry of the
            // tile is a candidate), before searching what is left
            if (hi - lo > 2) {
                const uint32_t g = lo + 1 + (uint32_t)((uint64_t)(x - t * kPTile) * (hi - lo - 1) /
                                                       kPTile);
                const uint32_t left = a.cidx[g - 1], here = a.cidx[g];
                if (left >= x) hi = g - 1;
                else if (here >= x) lo = hi = g;
                else lo = g + 1;
            }
        }
        while (lo < hi) {
            const uint32_t mid = (lo + hi) >> 1;
            if (a.cidx[mid] < x) lo = mid + 1; else hi = mid;
        }
        a.cand_off[s] = (s == a.nseg) ? total : lo;
    }
    __syncthreads();
    // the segments of every emit tile's first and last candidate, searched in a shared-memory
    // copy of the ranges when they fit
    const uint32_t etiles = (total + kEmitTile - 1) / kEmitTile;
    const bool staged = a.nseg < kCandoffStage;
    if (staged)
        for (int s = threadIdx.x; s <= a.nseg; s += blockDim.x) s_coff[s] = a.cand_off[s];
    __syncthreads();
    const uint32_t* co = staged ? s_coff : a.cand_off;
    for (uint32_t t = threadIdx.x; t < etiles; t += blockDim.x) {
        const uint32_t f0 = t * kEmitTile, f1 = (uint32_t)umin64(total, (uint64_t)f0 + kEmitTile) - 1u;
        a.eseg[2 * t] = (uint32_t)upper_bound_minus1(co, a.nseg, f0);
        a.eseg[2 * t + 1] = (uint32_t)upper_bound_minus1(co, a.nseg, f1);
    }
    uint32_t any_failed = 0, active = 0;
    for (int s = threadIdx.x; s < a.nseg; s += blockDim.x) {
        SegInfo& d = a.segs[s];
        const uint32_t cnt = a.cand_off[s + 1] - a.cand_off[s];
        d.cand_cnt = cnt;
        d.prefix = 0;
        d.state = kIdle;
        d.sel_x = 0;
        if (d.k == 0) continue;
        if (a.hp.mode == DGC_SELECT_EXACT) {
            if (cnt < d.k) {
                d.failed = 1;
                any_failed = 1;
            } else if (cnt > d.k) {
                d.state = kActive;
                d.need = d.k;
                ++active;
            }
        } else if (a.hp.mode == DGC_SELECT_SAMPLED &&
                   (unsigned __int128)cnt * kBillion > (unsigned __int128)a.hp.q_ppb * d.k) {
            d.resel = 1;
            d.state = kActive;
            d.need = d.k;
            ++active;
        }
    }
    if (active) atomicAdd(&s_active, active);
    if (any_failed) a.ctl->any_failed = 1;
    __syncthreads();
    if (threadIdx.x == 0) a.ctl->active = s_active;
}

// ---------------------------------------------------------------------------------- emit
// Candidates in index order; selected <=> X >= sel_x of their segment. Positions of the
// selected ones come from a decoupled look-back. Each sent entry leaves the accumulator
// (v <- 0) and, with masking, its momentum (u <- 0). The last block to finish writes out_count
// and the statistics.
__global__ void __launch_bounds__(kThreads) k_emit(Args a) {
    __shared__ uint32_t s_bitmap[kEmitTile / 32];
    __shared__ uint32_t s_wordpre[kEmitTile / 32];
    __shared__ uint32_t s_scan[33];
    __shared__ uint32_t s_tile;
    __shared__ uint64_t s_base;
    __shared__ int s_last, s_ok;
    if (threadIdx.x == 0) s_ok = !ld_relaxed_u32((const uint32_t*)&a.ctl->abort);
    __syncthreads();
    const bool ok = s_ok;
    const uint32_t total = a.ctl->total_cand;
    const bool unspec = ld_relaxed_u32(&a.ctl->unspec) != 0;
    const uint32_t ntiles = (total + kEmitTile - 1) / kEmitTile;
    while (ok) {
        if (threadIdx.x == 0) s_tile = atomicAdd(&a.ctl->ticket_emit, 1u);
        for (int w = threadIdx.x; w < kEmitTile / 32; w += kThreads) s_bitmap[w] = 0;
        __syncthreads();
        const uint32_t tile = s_tile;
        if (tile >= ntiles) break;
        const uint64_t base = (uint64_t)tile * kEmitTile;
        // the tile's candidates lie in segments [es0, es0 + ens) (from k_candoff): short searches
        const int es0 = (int)a.eseg[2 * tile], ens = (int)a.eseg[2 * tile + 1] - es0 + 1;
        uint32_t sel = 0;
        uint32_t idx[kEmitRows * 4];
        float val[kEmitRows * 4];
        int seg[kEmitRows * 4];
#pragma unroll
        for (int r = 0; r < kEmitRows; ++r) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint64_t i = base + 4u * (r * kThreads + threadIdx.x) + e;
                const int q = r * 4 + e;
                seg[q] = -1;
                if (i < total) {
                    idx[q] = a.cidx[i];
                    val[q] = a.cval[i];
                    const int s = es0 + upper_bound_minus1(a.cand_off + es0, ens, (uint32_t)i);
                    seg[q] = s;
                    const SegInfo& d = a.segs[s];
                    if (a.hp.bin) {  // AdaComp: the candidate reaches its bin's largest key
                        const uint32_t key = key_of(val[q]);
                        if (key > 0 && key == a.binmax[d.binbase + (idx[q] - d.start) / a.hp.bin])
                            sel |= 1u << q;
                    } else {
                        const uint64_t x = ((uint64_t)key_of(val[q]) << 32) | (uint64_t)(~idx[q]);
                        if (x >= d.sel_x) sel |= 1u << q;
                    }
                }
            }
            const uint32_t f4 = (sel >> (4 * r)) & 0xFu;
            if (f4) {
                const uint32_t off = 4u * (r * kThreads + threadIdx.x);
                atomicOr(&s_bitmap[off >> 5], f4 << (off & 31));
            }
        }
        __syncthreads();
        uint32_t cnt = 0;
        for (int w = threadIdx.x; w < kEmitTile / 32; w += kThreads) cnt += __popc(s_bitmap[w]);
        uint32_t tile_total;
        const uint32_t ex = block_excl_scan<kThreads>(cnt, s_scan, &tile_total);
        if (threadIdx.x < kEmitTile / 32) s_wordpre[threadIdx.x] = ex;
        if (threadIdx.x < 32) {
            const uint64_t excl = lookback_exclusive(a.st_emit, tile, tile_total, a.spin_limit,
                                                     a.status, &a.ctl->abort);
            if (threadIdx.x == 0) s_base = excl;
        }
        __syncthreads();
        const uint64_t gbase = s_base;
        int my_seg = -1;             // the smallest key sent and the number sent, per segment:
        uint32_t my_min = 0xFFFFFFFFu;  // one atomic per warp
        uint32_t my_cnt = 0;
#pragma unroll
        for (int q = 0; q < kEmitRows * 4; ++q) {
            if (seg[q] < 0) continue;
            const uint64_t i = base + 4u * ((q >> 2) * kThreads + threadIdx.x) + (q & 3);
            if (sel & (1u << q)) {
                const uint32_t key = key_of(val[q]);
                if (my_seg < 0) my_seg = seg[q];
                if (seg[q] == my_seg) {
                    my_min = min(my_min, key);
                    ++my_cnt;
                } else {
                    atomicMin(&a.segs[seg[q]].min_key, key);
                    atomicAdd(&a.segs[seg[q]].nsent, 1u);
                }
                const uint32_t off = (uint32_t)(i - base);
                const uint32_t w = off >> 5;
                const uint64_t pos =
                    gbase + s_wordpre[w] + __popc(s_bitmap[w] & ((1u << (off & 31)) - 1u));
                if (pos < a.out_cap) {
                    a.out_idx[pos] = idx[q];
                    a.out_val[pos] = val[q];
                }
                if (spec_slot(a, i, idx[q], total, unspec) < 0) {  // not yet stored as sent
                    a.v[idx[q]] = 0.0f;
                    if (a.hp.mask) a.u[idx[q]] = 0.0f;
                }
            } else {
                // a candidate the selection leaves out: put back what a speculative send stored
                const int64_t slot = spec_slot(a, i, idx[q], total, unspec);
                if (slot >= 0) {
                    a.v[idx[q]] = val[q];
                    if (a.hp.mask) a.u[idx[q]] = a.su[slot];
                }
            }
        }
        {
            const unsigned group = __match_any_sync(kFull, my_seg);
            const uint32_t gmin = __reduce_min_sync(group, my_min);
            const uint32_t gcnt = __reduce_add_sync(group, my_cnt);
            if (my_seg >= 0 && (threadIdx.x & 31) == __ffs(group) - 1) {
                atomicMin(&a.segs[my_seg].min_key, gmin);
                atomicAdd(&a.segs[my_seg].nsent, gcnt);
            }
        }
        if (tile == ntiles - 1 && threadIdx.x == 0) a.ctl->total_sent = (uint32_t)(gbase + tile_total);
        __syncthreads();
    }
    // the last block out writes the results
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(&a.ctl->emit_done, 1u) == gridDim.x - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x == 0 && ok) *a.out_count = (int64_t)ld_relaxed_u32(&a.ctl->total_sent);
    if (!a.stats) return;
    for (int s = threadIdx.x; s < a.nseg; s += kThreads) {
        const SegInfo& d = a.segs[s];
        dgc_seg_stats o;
        o.k = d.k;
        uint64_t sent = 0;
        if (ok && d.k > 0) {
            if (a.hp.mode == DGC_SELECT_EXACT) sent = d.k;
            else if (a.hp.mode == DGC_SELECT_ADACOMP) sent = ld_relaxed_u32(&d.nsent);
            else sent = d.resel ? d.k : d.cand_cnt;
        }
        o.sent = sent;
        o.candidates = (a.hp.mode != DGC_SELECT_SAMPLED) ? sent : (ok ? d.cand_cnt : 0);
        o.thresh_key = ld_relaxed_u32(&d.min_key);
        o.sample_key = (a.hp.mode == DGC_SELECT_SAMPLED && d.k > 0) ? d.thresh : 0u;
        o.reselected = d.resel;
        o.clip_scale = d.scale;
        o.clip_sumsq = d.sumsq;
        a.stats[s] = o;
    }
}

// ------------------------------------------------------------------ shared index set
// A learner that sends at an index set chosen elsewhere (one set for all learners, so their
// messages add up position by position). The set is checked before anything changes: strictly
// ascending, below n, and count within [0, max_count]; otherwise the call reports DGC_EINVAL and
// the abort flag stops every later kernel of the call.
__global__ void __launch_bounds__(kThreads) k_shared_check(Args a, const uint32_t* idx,
                                                          const int64_t* count,
                                                          uint64_t max_count) {
    const int64_t c = *count;
    if (c < 0 || (uint64_t)c > max_count) {
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            report(a.status, DGC_EINVAL);
            atomicExch(&a.ctl->abort, 1);
        }
        return;
    }
    bool bad = false;
    for (uint64_t j = (uint64_t)blockIdx.x * kThreads + threadIdx.x; j < (uint64_t)c;
         j += (uint64_t)gridDim.x * kThreads)
        if (idx[j] >= a.n || (j > 0 && idx[j - 1] >= idx[j])) bad = true;
    if (__syncthreads_or(bad) && threadIdx.x == 0) {
        report(a.status, DGC_EINVAL);
        atomicExch(&a.ctl->abort, 1);
    }
}

// After the accumulate-only pass: out_val[j] = v[idx[j]], then the entry leaves the accumulator
// (v <- 0; u <- 0 with momentum factor masking).
__global__ void __launch_bounds__(kThreads) k_shared_gather(Args a, const uint32_t* idx,
                                                           const int64_t* count, float* out_val) {
    if (ld_relaxed_u32((const uint32_t*)&a.ctl->abort)) return;
    const uint64_t c = (uint64_t)*count;
    for (uint64_t j = (uint64_t)blockIdx.x * kThreads + threadIdx.x; j < c;
         j += (uint64_t)gridDim.x * kThreads) {
        const uint32_t i = idx[j];
        out_val[j] = a.v[i];
        a.v[i] = 0.0f;
        if (a.hp.mask) a.u[i] = 0.0f;
    }
}

}  // namespace
}  // namespace dgc

using namespace dgc;

static cudaEvent_t g_prof_begin = nullptr, g_prof_end = nullptr;

// A profiling marker on the call's stream. Under stream capture it becomes an event-record node
// of the graph, so every launch of the graph records it.
static void record_marker(cudaEvent_t ev, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
    else
        cudaEventRecord(ev, s);
}

extern "C" void dgc_profile_stream_pass(dgc_event_t begin, dgc_event_t end) {
    g_prof_begin = reinterpret_cast<cudaEvent_t>(begin);
    g_prof_end = reinterpret_cast<cudaEvent_t>(end);
}

extern "C" int dgc_compress_workspace(int64_t n, int32_t nseg, const dgc_params* params,
                                      size_t* bytes) {
    HostParams hp{};
    if (!bytes || nseg < 1 || n < 0) return DGC_EINVAL;
    if (n > 0xFFFFFFFFll || nseg > (1 << 28)) return DGC_EUNSUPPORTED;
    const int rc = check_params(params, &hp);
    if (rc) return rc;
    *bytes = make_layout(n, nseg, hp).total;
    return DGC_OK;
}

extern "C" int dgc_compress_max_out(int64_t n, int32_t nseg, const dgc_params* params,
                                    int64_t* max_out) {
    HostParams hp{};
    if (!max_out || nseg < 1 || n < 0) return DGC_EINVAL;
    if (n > 0xFFFFFFFFll || nseg > (1 << 28)) return DGC_EUNSUPPORTED;
    const int rc = check_params(params, &hp);
    if (rc) return rc;
    *max_out = (int64_t)max_out_for(n, nseg, hp);
    return DGC_OK;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

namespace dgc {
namespace {
// The kernels' view of one call: caller buffers and the workspace carved by the layout L.
Args make_args(const float* g, float* u, float* v, int64_t n, const int64_t* seg_off,
               int32_t nseg, const HostParams& hp, const Layout& L, void* ws, int32_t* status) {
    char* w = static_cast<char*>(ws);
    Args a{};
    a.g = g;
    a.u = u;
    a.v = v;
    a.n = (uint32_t)n;
    a.nseg = nseg;
    a.seg_off = seg_off;
    a.hp = hp;
    a.status = status;
    a.ctl = reinterpret_cast<Ctl*>(w + L.ctl);
    a.scache = reinterpret_cast<SampleCache*>(w + L.scache);
    a.segs = reinterpret_cast<SegInfo*>(w + L.segs);
    a.seg_start = reinterpret_cast<uint32_t*>(w + L.seg_start);
    a.samp_off = reinterpret_cast<uint32_t*>(w + L.samp_off);
    a.clip_off = reinterpret_cast<uint32_t*>(w + L.clip_off);
    a.cand_off = reinterpret_cast<uint32_t*>(w + L.cand_off);
    a.clip_acc = reinterpret_cast<unsigned long long*>(w + L.clip_acc);
    a.skeys = reinterpret_cast<uint32_t*>(w + L.skeys);
    a.spos = reinterpret_cast<uint32_t*>(w + L.spos);
    a.bcount = reinterpret_cast<uint32_t*>(w + L.bcount);
    a.histA = reinterpret_cast<uint32_t*>(w + L.histA);
    a.histB = reinterpret_cast<uint32_t*>(w + L.histB);
    a.st_collect = reinterpret_cast<uint64_t*>(w + L.st_collect);
    a.st_compact = reinterpret_cast<uint64_t*>(w + L.st_compact);
    a.st_emit = reinterpret_cast<uint64_t*>(w + L.st_emit);
    a.cidx = reinterpret_cast<uint32_t*>(w + L.cidx);
    a.sidx = reinterpret_cast<uint32_t*>(w + L.sidx);
    a.cval = reinterpret_cast<float*>(w + L.sidx);
    a.sval = reinterpret_cast<float*>(w + L.sval);
    a.su = reinterpret_cast<float*>(w + L.su);
    a.tcount = reinterpret_cast<uint32_t*>(w + L.tcount);
    a.tseg = reinterpret_cast<uint32_t*>(w + L.tseg);
    a.eseg = reinterpret_cast<uint32_t*>(w + L.eseg);
    a.clip_cnt = reinterpret_cast<uint32_t*>(w + L.clip_cnt);
    a.dlist = reinterpret_cast<uint32_t*>(w + L.dlist);
    a.binmax = reinterpret_cast<uint32_t*>(w + L.binmax);
    a.max_samples = L.max_samples;
    a.fused_tiles = L.fused_tiles;
    a.ptiles = L.ptiles;
    a.cgroups = L.cgroups;
    a.nbuckets = L.nbuckets;
    a.max_bins = L.max_bins;
    a.emit_tiles = L.emit_tiles;
    a.max_clip_tiles = L.max_clip_tiles;
    a.spin_limit = kDefaultSpinLimit;
    return a;
}

template <int kSel>
void stream_attributes() {
    cudaFuncSetAttribute(k_stream_tma<kSel>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)stream_smem_bytes<kSel>());
    // the AdaComp variant needs nearly all of the SM's shared memory for two blocks
    cudaFuncSetAttribute(k_stream_tma<kSel>, cudaFuncAttributePreferredSharedMemoryCarveout,
                         (int)cudaSharedmemCarveoutMaxShared);
}

// Shared-memory limits of the kernels that need more than 48 KiB, once per device.
void set_kernel_attributes() {
    static bool attr_set[128] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 128 && !attr_set[dev]) {
        stream_attributes<0>();
        stream_attributes<1>();
        stream_attributes<2>();
        cudaFuncSetAttribute(k_select_small<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmallBytes);
        cudaFuncSetAttribute(k_select_small<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmallBytes);
        cudaFuncSetAttribute(k_clip_tiles, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kClipSmem);
        attr_set[dev] = true;
    }
}

// Blocks of a cooperative launch (0, 1: the global select of sample keys / candidates; 2: the
// sample-position cache): all resident at once, up to 4 per SM (more loads in flight over the
// items); the occupancy is asked once per device.
unsigned cooperative_grid(int which, int sms) {
    static int per_sm[3][128] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    int b = (dev >= 0 && dev < 128) ? per_sm[which][dev] : 0;
    if (b == 0) {
        if (which == 0)
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_select_global<0>, kThreads, 0);
        else if (which == 1)
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_select_global<1>, kThreads, 0);
        else
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_cache, kThreads, 0);
        b = std::max(1, std::min(4, b));
        if (dev >= 0 && dev < 128) per_sm[which][dev] = b;
    }
    return (unsigned)(b * sms);
}

// The streaming pass: persistent blocks, 2 or 3 per SM (at most one per tile).
void launch_stream_pass(int sel, const Args& a, uint64_t ptiles, int sms, cudaStream_t s) {
    set_kernel_attributes();
    auto grid = [&](int per_sm) {
        return (unsigned)std::min<uint64_t>((uint64_t)sms * per_sm, ptiles);
    };
    if (sel == 1)
        k_stream_tma<1><<<grid(stream_blocks_per_sm<1>()), kThreads, stream_smem_bytes<1>(), s>>>(a);
    else if (sel == 2)
        k_stream_tma<2><<<grid(stream_blocks_per_sm<2>()), kThreads, stream_smem_bytes<2>(), s>>>(a);
    else
        k_stream_tma<0><<<grid(stream_blocks_per_sm<0>()), kThreads, stream_smem_bytes<0>(), s>>>(a);
}
}  // namespace
}  // namespace dgc

extern "C" int dgc_compress(const float* g, float* u, float* v, int64_t n, const int64_t* seg_off,
                            int32_t nseg, const dgc_params* params, uint32_t* out_idx,
                            float* out_val, int64_t out_cap, int64_t* out_count,
                            dgc_seg_stats* stats, int32_t* status, void* ws, size_t ws_bytes,
                            dgc_stream_t stream) {
    HostParams hp{};
    if (n < 0 || nseg < 1) return DGC_EINVAL;
    if (n > 0xFFFFFFFFll || nseg > (1 << 28)) return DGC_EUNSUPPORTED;
    int rc = check_params(params, &hp);
    if (rc) return rc;
    if (!seg_off || !out_count || !status || !ws) return DGC_EINVAL;
    if (n > 0 && (!g || !u || !v || !aligned16(g) || !aligned16(u) || !aligned16(v)))
        return DGC_EINVAL;
    if (((uintptr_t)ws & 255u) != 0) return DGC_EINVAL;
    const Layout L = make_layout(n, nseg, hp);
    if (ws_bytes < L.total) return DGC_EINVAL;
    const uint64_t mo = max_out_for(n, nseg, hp);
    if (out_cap < 0 || (uint64_t)out_cap < mo) return DGC_ECAPACITY;
    if (mo > 0 && (!out_idx || !out_val)) return DGC_EINVAL;

    Args a = make_args(g, u, v, n, seg_off, nseg, hp, L, ws, status);
    a.out_idx = out_idx;
    a.out_val = out_val;
    a.out_cap = (uint64_t)out_cap;
    a.out_count = out_count;
    a.stats = stats;

    const int sms = dgc_internal_sm_count();
    if (sms <= 0) return DGC_ECUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint64_t launches = 0;
    auto L1 = [&](auto kernel, unsigned grid, unsigned block, auto... args) {
        if (grid == 0) return;
        kernel<<<grid, block, 0, s>>>(args...);
        ++launches;
    };
    const size_t zero_work = (size_t)nseg * kHistBins + L.fused_tiles + L.emit_tiles +
                             L.nbuckets + L.max_bins + L.ptiles + 3;
    const unsigned plan_grid = (unsigned)std::min<size_t>((zero_work + 1023) / 1024 + 1,
                                                          (size_t)sms * 2);
    set_kernel_attributes();  // before the first launch that needs more than 48 KiB
    L1(k_plan, plan_grid, 1024, a);
    if (hp.clip_on) {
        k_clip_tiles<<<(unsigned)std::max<uint64_t>(
                           1, std::min<uint64_t>(L.max_clip_tiles, (uint64_t)sms * 4)),
                       kThreads, kClipSmem, s>>>(a);
        ++launches;
        L1(k_clip_round, (unsigned)((nseg + 127) / 128), 128, a);
    }
    bool launch_failed = false;
    auto coop = [&](const void* kernel, unsigned grid) {
        void* args[] = {&a};
        if (cudaLaunchCooperativeKernel(kernel, dim3(grid), dim3(kThreads), args, 0, s) !=
            cudaSuccess)
            launch_failed = true;
        ++launches;
    };
    // AdaComp draws no sample and keeps every segment idle: no cache, sample or select launches
    const bool selects = hp.mode != DGC_SELECT_ADACOMP;
    if (selects) {
        coop((const void*)k_cache, cooperative_grid(2, sms));
        const uint64_t sgrid = (L.max_samples + kThreads * kSamplePerThread - 1) /
                               (kThreads * kSamplePerThread);
        L1(k_sample, (unsigned)sgrid, kThreads, a);
    }
    set_kernel_attributes();
    auto global_select = [&](int kind) {
        coop(kind == 0 ? (const void*)k_select_global<0> : (const void*)k_select_global<1>,
             cooperative_grid(kind, sms));
    };
    auto small_select = [&](int kind) {
        if (kind == 0)
            k_select_small<0><<<(unsigned)nseg, kSmallThreads, kSmallBytes, s>>>(a);
        else
            k_select_small<1><<<(unsigned)nseg, kSmallThreads, kSmallBytes, s>>>(a);
        ++launches;
    };
    if (selects) {
        small_select(0);
        global_select(0);
    }
    const cudaEvent_t pb = g_prof_begin, pe = g_prof_end;
    if (pb && pe) record_marker(pb, s);
    if (n > 0) {
        launch_stream_pass(hp.mode == DGC_SELECT_ADACOMP ? 1 : 0, a, L.ptiles, sms, s);
        ++launches;
    }
    if (pb && pe) record_marker(pe, s);
    L1(k_collect, (unsigned)L.cgroups, kThreads, a);
    L1(k_collect_copy, (unsigned)sms * 8, kThreads, a);
    L1(k_candoff, 1, 1024, a, 0);
    if (hp.mode == DGC_SELECT_EXACT) {
        L1(k_unspec, (unsigned)sms * 8, kThreads, a);
        L1(k_recompact, (unsigned)L.fused_tiles, kThreads, a);
        L1(k_candoff, 1, 1024, a, 1);
    }
    L1(k_cval, (unsigned)sms * 8, kThreads, a);
    if (selects) {
        small_select(1);
        global_select(1);
    }
    const unsigned emit_grid = (unsigned)std::max<uint64_t>(
        1, std::min<uint64_t>((uint64_t)sms * 4, L.emit_tiles));
    L1(k_emit, emit_grid, kThreads, a);
    dgc_internal_count_launches(launches);
    if (launch_failed || cudaPeekAtLastError() != cudaSuccess) {
        cudaGetLastError();
        return DGC_ECUDA;
    }
    return DGC_OK;
}

extern "C" int dgc_compress_shared(const float* g, float* u, float* v, int64_t n,
                                   const int64_t* seg_off, int32_t nseg, const dgc_params* params,
                                   const uint32_t* idx, const int64_t* count, int64_t max_count,
                                   float* out_val, int32_t* status, void* ws, size_t ws_bytes,
                                   dgc_stream_t stream) {
    HostParams hp{};
    if (n < 0 || nseg < 1 || max_count < 0) return DGC_EINVAL;
    if (n > 0xFFFFFFFFll || nseg > (1 << 28)) return DGC_EUNSUPPORTED;
    int rc = check_params(params, &hp);
    if (rc) return rc;
    // no selection: every segment's k is 0, so the plan draws no sample and counts no bin
    hp.mode = DGC_SELECT_EXACT;
    hp.d_ppb = 0;
    hp.bin = 0;
    hp.nospec = 1;
    if (!seg_off || !count || !status || !ws) return DGC_EINVAL;
    if (max_count > 0 && (!idx || !out_val)) return DGC_EINVAL;
    if (n > 0 && (!g || !u || !v || !aligned16(g) || !aligned16(u) || !aligned16(v)))
        return DGC_EINVAL;
    if (((uintptr_t)ws & 255u) != 0) return DGC_EINVAL;
    const Layout L = make_layout(n, nseg, hp);
    if (ws_bytes < L.total) return DGC_EINVAL;
    Args a = make_args(g, u, v, n, seg_off, nseg, hp, L, ws, status);
    a.out_count = nullptr;  // the count is the caller's input here

    const int sms = dgc_internal_sm_count();
    if (sms <= 0) return DGC_ECUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint64_t launches = 0;
    auto L1 = [&](auto kernel, unsigned grid, unsigned block, auto... args) {
        if (grid == 0) return;
        kernel<<<grid, block, 0, s>>>(args...);
        ++launches;
    };
    const size_t zero_work = (size_t)nseg * kHistBins + L.fused_tiles + L.emit_tiles +
                             L.nbuckets + L.max_bins + L.ptiles + 3;
    const unsigned plan_grid = (unsigned)std::min<size_t>((zero_work + 1023) / 1024 + 1,
                                                          (size_t)sms * 2);
    const unsigned jgrid = (unsigned)std::max<uint64_t>(
        1, std::min<uint64_t>((uint64_t)sms * 4, ((uint64_t)max_count + kThreads - 1) / kThreads));
    set_kernel_attributes();  // before the first launch that needs more than 48 KiB
    L1(k_plan, plan_grid, 1024, a);
    L1(k_shared_check, jgrid, kThreads, a, idx, count, (uint64_t)max_count);
    if (hp.clip_on) {
        k_clip_tiles<<<(unsigned)std::max<uint64_t>(
                           1, std::min<uint64_t>(L.max_clip_tiles, (uint64_t)sms * 4)),
                       kThreads, kClipSmem, s>>>(a);
        ++launches;
        L1(k_clip_round, (unsigned)((nseg + 127) / 128), 128, a);
    }
    const cudaEvent_t pb = g_prof_begin, pe = g_prof_end;
    if (pb && pe) record_marker(pb, s);
    if (n > 0) {
        launch_stream_pass(2, a, L.ptiles, sms, s);
        ++launches;
    }
    if (pb && pe) record_marker(pe, s);
    L1(k_shared_gather, jgrid, kThreads, a, idx, count, out_val);
    dgc_internal_count_launches(launches);
    if (cudaPeekAtLastError() != cudaSuccess) {
        cudaGetLastError();
        return DGC_ECUDA;
    }
    return DGC_OK;
}
