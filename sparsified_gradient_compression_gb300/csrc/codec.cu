// codec.cu -- dgc_encode, dgc_decode_accumulate and dgc_decode_apply on sm_103a.
//
// Source: "[Paper Review] Deep Gradient Compression: Reducing the Communication Bandwidth for
// Distributed Training", Proposed method, bullet 2 (each sent value as a 32-bit word and the
// run of zeros before it as a 16-bit length), and Abstract / Motivation (synchronous SGD adds
// up the learners' updates). Byte layout (this library's reading): 32-byte header
// ("DGC1", u16 version 1, u16 flags 0, u64 n, u64 T, u64 nnz), T binary32 values, T u16 runs,
// zero pad to a multiple of 4; a run of 0xFFFF is an escape that skips 65535 zeros.
//
// Encode: reduce-then-scan over the (ascending) entries. Block b owns a contiguous share; pass
// 1 counts its tokens (1 + gap/65535 per entry), one block scans the G totals and writes the
// header, pass 2 writes values and runs at their final offsets.
//
// Decode: pass 1 turns each message's runs into positions with a prefix sum over 2048-token
// chunks (decoupled look-back inside each message) and records, for every 4096-entry tile of
// the dense output, the first token of each message at or past the tile. Pass 2 gives each
// tile to one block: it gathers the tile's tokens of all messages into shared memory, adds them
// in message order 0..W-1 into a shared-memory copy of the tile, and writes the tile once. Each
// dense entry is therefore written exactly once and summed in a fixed order.
//
// Decode-apply (dgc_decode_apply) runs the same passes but never materialises the dense sum:
// each tile's sum, built from +0 in the same order, updates the weights w <- fma(-lr, sum, w)
// only where a message landed (elsewhere the update is the identity), so w is read and written
// at the touched positions instead of streaming a dense array through HBM.
#include <cmath>
#include <vector>

#include "dgc_device.cuh"

namespace dgc {
namespace {

constexpr int kThreads = 256;
constexpr int kEncBlocks = 512;
constexpr int kEncPer = 4;
constexpr int kDecChunk = 4096;  // tokens per position chunk
constexpr int kPosThreads = 256; // threads of the position kernel (16 tokens each)
constexpr int kDecTile = 4096;   // dense entries per output tile
constexpr int kDecCap = 512;     // tokens staged in shared memory at a time
constexpr uint32_t kEscPos = 0xFFFFFFFFu;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ------------------------------------------------------------------------------ encode
// Written by the scan kernel alone (no clearing before the call): whether the call stops before
// the write, and the token count.
struct EncCtl {
    int32_t abort;
    uint32_t pad;
    uint64_t T;
};

struct EncArgs {
    const uint32_t* idx;
    const float* val;
    const int64_t* count;
    uint64_t max_count;
    uint64_t n;
    uint8_t* out;
    uint64_t out_cap;
    uint64_t* out_bytes;
    int32_t* status;
    EncCtl* ctl;
    uint64_t* tot;  // per-block token counts, then exclusive offsets
    int32_t qbits;  // 0: binary32 values (version 1); 8 or 16: integers (version 2)
    float alpha;    // version 2: the shared scale
    float* v;       // version 2: residual that takes back what the integers do not carry
};

// Programmatic dependent launch: a kernel launched with programmatic stream serialization may
// start before the kernel ahead of it in the stream has finished; it waits here before it reads
// anything that kernel writes (a no-op when it was launched the ordinary way). The kernel ahead
// lets its dependents launch as soon as each of its blocks has started.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// version 2 layout: values of qbits/8 bytes, runs from the next even offset, nothing after them
// (so the size fixes T: the receiver lays the messages out from their sizes)
__host__ __device__ __forceinline__ uint64_t q_runs_offset(uint64_t T, int qbits) {
    const uint64_t at = 32 + T * (uint64_t)(qbits / 8);
    return at + (at & 1);
}
__host__ __device__ __forceinline__ uint64_t q_size(uint64_t T, int qbits) {
    return q_runs_offset(T, qbits) + 2 * T;
}

// q = clamp(rint(alpha * x), -Q, Q); the conversion rounds half to even and takes NaN to 0
__device__ __forceinline__ int32_t quantize(float x, float alpha, int qbits) {
    const int32_t Q = (1 << (qbits - 1)) - 1;
    const int32_t q = __float2int_rn(__fmul_rn(alpha, x));
    return q > Q ? Q : (q < -Q ? -Q : q);
}

__device__ __forceinline__ bool enc_range(const EncArgs& a, uint64_t* lo, uint64_t* hi,
                                          uint64_t* cnt) {
    const int64_t c = *a.count;
    if (c < 0 || (uint64_t)c > a.max_count) return false;
    *cnt = (uint64_t)c;
    const uint64_t per = ((uint64_t)c + gridDim.x - 1) / gridDim.x;
    *lo = umin64((uint64_t)c, (uint64_t)blockIdx.x * per);
    *hi = umin64((uint64_t)c, *lo + per);
    return true;
}

__device__ __forceinline__ uint64_t enc_tokens(const EncArgs& a, uint64_t j, bool* bad) {
    const int64_t cur = a.idx[j];
    const int64_t prev = j ? (int64_t)a.idx[j - 1] : -1;
    if ((uint64_t)cur >= a.n || cur <= prev) {
        *bad = true;
        return 1;
    }
    return 1 + (uint64_t)(cur - prev - 1) / kRunEscape;
}

// a block's token count that marks an index out of range or out of order
constexpr uint64_t kTotBad = ~0ull;

__global__ void __launch_bounds__(kThreads) k_enc_count(EncArgs a) {
    __shared__ uint64_t s_scan[33];
    __shared__ int s_bad;
    grid_dep_launch();
    uint64_t lo, hi, cnt;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    if (!enc_range(a, &lo, &hi, &cnt)) {  // (the scan kernel finds the count bad as well)
        if (blockIdx.x == 0 && threadIdx.x == 0) report(a.status, DGC_EINVAL);
        return;
    }
    uint64_t t = 0;
    bool bad = false;
    for (uint64_t j = lo + threadIdx.x; j < hi; j += kThreads) t += enc_tokens(a, j, &bad);
    if (bad) s_bad = 1;
    uint64_t total;
    block_excl_scan<kThreads>(t, s_scan, &total);
    if (threadIdx.x == 0) {
        a.tot[blockIdx.x] = s_bad ? kTotBad : total;
        if (s_bad) report(a.status, DGC_EINVAL);
    }
}

__global__ void __launch_bounds__(1024) k_enc_scan(EncArgs a, int nblocks) {
    __shared__ uint64_t s_scan[33];
    grid_dep_launch();
    grid_dep_wait();
    // a count out of range, or a block that found a bad index: no message (the count kernel
    // reported it)
    const int64_t c = *a.count;
    const bool count_ok = c >= 0 && (uint64_t)c <= a.max_count;
    const uint64_t x = (count_ok && threadIdx.x < nblocks) ? a.tot[threadIdx.x] : 0;
    if (__syncthreads_or(!count_ok || x == kTotBad)) {
        if (threadIdx.x == 0) {
            *a.out_bytes = 0;
            a.ctl->abort = 1;
        }
        return;
    }
    uint64_t T;
    const uint64_t ex = block_excl_scan<1024>(x, s_scan, &T);
    if (threadIdx.x < nblocks) a.tot[threadIdx.x] = ex;
    if (threadIdx.x != 0) return;
    const uint64_t bytes = a.qbits ? q_size(T, a.qbits) : 32 + 6 * T + ((T & 1) ? 2 : 0);
    *a.out_bytes = bytes;
    if (bytes > a.out_cap) {
        report(a.status, DGC_ECAPACITY);
        a.ctl->abort = 1;
        return;
    }
    a.ctl->T = T;
    a.ctl->abort = 0;
    uint64_t* h = reinterpret_cast<uint64_t*>(a.out);
    h[1] = a.n;
    h[2] = T;
    if (a.qbits) {  // magic, version 2, width; alpha and the entry count share the last word
        h[0] = (uint64_t)kMagic | (2ull << 32) | ((uint64_t)a.qbits << 48);
        h[3] = (uint64_t)__float_as_uint(a.alpha) | ((uint64_t)*a.count << 32);
        const uint64_t vend = 32 + T * (uint64_t)(a.qbits / 8);
        if (vend & 1) a.out[vend] = 0;  // the pad byte before the runs
    } else {
        h[0] = (uint64_t)kMagic | (1ull << 32);  // magic, version 1, flags 0
        h[3] = (uint64_t)*a.count;
        if (T & 1) *reinterpret_cast<uint16_t*>(a.out + 32 + 6 * T) = 0;
    }
}

__global__ void __launch_bounds__(kThreads) k_enc_write(EncArgs a) {
    __shared__ uint64_t s_scan[33];
    uint64_t lo, hi, cnt;
    if (!enc_range(a, &lo, &hi, &cnt)) return;  // (the scan kernel stopped the call)
    uint32_t* vals = reinterpret_cast<uint32_t*>(a.out + 32);
    int8_t* vals8 = reinterpret_cast<int8_t*>(a.out + 32);
    int16_t* vals16 = reinterpret_cast<int16_t*>(a.out + 32);
    uint16_t* runs = nullptr;
    uint64_t carry = 0;
    bool waited = false;  // (the same in every thread)
    for (uint64_t c = lo; c < hi; c += (uint64_t)kThreads * kEncPer) {
        uint64_t tk[kEncPer];
        uint64_t mine = 0;
        bool bad = false;
#pragma unroll
        for (int e = 0; e < kEncPer; ++e) {
            const uint64_t j = c + (uint64_t)threadIdx.x * kEncPer + e;
            tk[e] = (j < hi) ? enc_tokens(a, j, &bad) : 0;
            mine += tk[e];
        }
        uint64_t total;
        const uint64_t ex = block_excl_scan<kThreads>(mine, s_scan, &total);
        if (!waited) {
            // the block's first tokens are counted (from inputs that came before the call) while
            // the scan kernel finishes; its results from here on
            grid_dep_wait();
            if (ld_relaxed_u32(reinterpret_cast<const uint32_t*>(&a.ctl->abort))) return;
            const uint64_t T = a.ctl->T;
            runs = reinterpret_cast<uint16_t*>(
                a.out + (a.qbits ? q_runs_offset(T, a.qbits) : 32 + 4 * T));
            carry = a.tot[blockIdx.x];
            waited = true;
        }
        uint64_t p = carry + ex;
#pragma unroll
        for (int e = 0; e < kEncPer; ++e) {
            const uint64_t j = c + (uint64_t)threadIdx.x * kEncPer + e;
            if (j >= hi) break;
            const int64_t prev = j ? (int64_t)a.idx[j - 1] : -1;
            const uint64_t gap = (uint64_t)((int64_t)a.idx[j] - prev - 1);
            for (uint64_t x = 1; x < tk[e]; ++x, ++p) {
                if (a.qbits == 8) vals8[p] = 0;
                else if (a.qbits == 16) vals16[p] = 0;
                else vals[p] = 0u;
                runs[p] = (uint16_t)kRunEscape;
            }
            const float x = a.val[j];
            if (a.qbits) {
                const int32_t q = quantize(x, a.alpha, a.qbits);
                if (a.qbits == 8) vals8[p] = (int8_t)q;
                else vals16[p] = (int16_t)q;
                if (a.v)  // the residual keeps x - q / alpha
                    a.v[a.idx[j]] = __fsub_rn(x, __fdiv_rn(__int2float_rn(q), a.alpha));
            } else {
                vals[p] = __float_as_uint(x);
            }
            runs[p] = (uint16_t)(gap % kRunEscape);
            ++p;
        }
        carry += total;
    }
}

// tokens of a message of `bytes` bytes; false when no message of that kind has that size
__host__ __device__ inline bool stream_tokens(uint64_t bytes, int qbits, uint64_t* T) {
    if (bytes < 32) return false;
    if (!qbits) {
        const uint64_t t = (bytes - 32) / 6;
        if (32 + 6 * t + ((t & 1) ? 2 : 0) != bytes) return false;
        *T = t;
        return true;
    }
    const uint64_t per = (uint64_t)qbits / 8 + 2;  // bytes per token; padding adds at most 4
    const uint64_t t0 = (bytes - 32) / per;
    for (uint64_t t = t0 > 2 ? t0 - 2 : 0; t <= t0; ++t)
        if (q_size(t, qbits) == bytes) {
            *T = t;
            return true;
        }
    return false;
}

// ------------------------------------------------------------------------------ decode
struct DecStream {
    const uint8_t* ptr;
    uint64_t T;
    uint64_t tok_base;
    uint64_t chunk_base;
    uint64_t runs_off;  // byte offset of the runs block
};

struct DecCtl {
    uint32_t any_bad;
    uint32_t pad;
};

struct DecArgs {
    DecStream* tab;  // W + 1 entries (the last holds the totals), in the workspace
    int32_t W;
    uint64_t n;
    float* dense;      // the dense sum, or the weights w when apply is set
    int32_t accumulate;
    int32_t apply;     // w <- fma(neg_lr, sum, w) at every position a message touches
    float neg_lr;
    int32_t qbits;     // 0: binary32 messages; 8 or 16: integer messages (version 2)
    float alpha;       // version 2: the shared scale every message must carry
    int32_t* status;
    DecCtl* ctl;
    uint32_t* pos;
    uint64_t* st;
    uint32_t* ts;  // (ntiles + 1) x W first-token table
    const uint64_t* dev_bytes;  // the message sizes in device memory, or null (sizes on the host)
    uint64_t ntiles;
    uint64_t nchunks;
    uint32_t spin_limit;
};

__device__ __forceinline__ void mark_bad(const DecArgs& a) {
    atomicExch(&a.ctl->any_bad, 1u);
    report(a.status, DGC_ECORRUPT);
}

// The message table by value, for calls with at most kDecInline messages: it travels with the
// launch (W + 1 entries within the 4 KB of kernel parameters), so no host memory is read when
// the call replays from a CUDA graph. Larger calls copy the table to the workspace instead.
constexpr int kDecInline = 96;
template <int kMax>
struct DecTabInline {
    DecStream e[kMax + 1];
};
static_assert(sizeof(DecTabInline<kDecInline>) + sizeof(DecArgs) <= 4096,
              "within the kernel parameter space");

// A message's header: magic, version, n and T (version 2: also the receiver's width and
// alpha, bit for bit).
__device__ bool header_ok(const DecArgs& a, const DecStream& d) {
    const uint64_t* h = reinterpret_cast<const uint64_t*>(d.ptr);
    const uint64_t h0 = h[0];
    bool ok = (uint32_t)h0 == kMagic && h[1] == a.n && h[2] == d.T;
    if (a.qbits)
        ok = ok && ((h0 >> 32) & 0xFFFFu) == 2u && (h0 >> 48) == (uint64_t)a.qbits &&
             (uint32_t)h[3] == __float_as_uint(a.alpha);
    else
        ok = ok && ((h0 >> 32) & 0xFFFFu) == 1u;
    return ok;
}

// Token positions, one chunk of kDecChunk tokens of one message per block (16 contiguous tokens
// per thread), in two launches. Token j advances the running position by run + 1 (an escape by
// 65535) and sits at the position the advance reaches, less one. The first launch (kPass 0) sums
// each chunk's advances and publishes the sum in the chunk's look-back word; the second (kPass
// 1) finds every word of a chunk's predecessors already written, so its look-back over them
// reads and never waits (within one launch a chunk's look-back waited microseconds for words
// its predecessors had written already). Within the chunk every sum is taken in 32 bits (a chunk
// advances by less than 2^28); the chunk's base, from the look-back, in 64 bits. Each token's
// end e = position + 1 is checked against n once; e <= n makes the 32-bit position exact. A
// token is the first of its message in the tiles t with e_prev <= t kDecTile < e (e_prev the
// previous token's end, 0 before the first), and the message's last token also fills the table
// for every later tile.
//
// Every message owns at least one chunk. In the first launch the block of its first chunk writes
// its entry of the workspace table for the kernels that follow (with the token count read from
// device memory when the sizes are there) and, for a message without tokens, fills the message's
// column of the first-token table with 0; block 0 clears the call's control word. The second
// launch may start while the first finishes: it reads its chunk's runs and scans them, then
// waits for the first launch before the look-back, and its first-chunk blocks check the headers
// (so every mark of a malformed message comes after the clear). The look-back words need no
// clearing: a chunk reads only the words of its own message's earlier chunks, all written by the
// first launch of the same call.
template <int kMax, int kPass>
__global__ void __launch_bounds__(kPosThreads, 1024 / kPosThreads)
    k_dec_pos(DecArgs a, const __grid_constant__ DecTabInline<kMax> t) {
    __shared__ uint32_t s_scan[33];
    __shared__ uint64_t s_lb64[33];
    __shared__ uint32_t s_lb32[2];
    __shared__ uint64_t s_cb[kPosThreads];  // the messages' first chunks, when W <= kPosThreads
    grid_dep_launch();  // the next launch may start once every block here has
    // the host's table: with the launch (up to kMax messages), else copied to the workspace
    const DecStream* tin = (a.W <= kMax) ? t.e : a.tab;
    const bool staged = a.W <= kPosThreads;
    if (staged && threadIdx.x < a.W) s_cb[threadIdx.x] = tin[threadIdx.x].chunk_base;
    __syncthreads();
    const uint64_t c = blockIdx.x;
    // the message that owns chunk c: the last one starting at or before c, searched in shared
    // memory (one parallel load instead of a chain of them)
    int lo = 0, hi = a.W;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((staged ? s_cb[mid] : tin[mid].chunk_base) <= c) lo = mid; else hi = mid;
    }
    const int w = lo;
    DecStream d = tin[w];
    bool size_ok = true;
    if (a.dev_bytes) {
        // sizes in device memory: the table holds each message's bound on T (from its bound on
        // bytes); the real T comes from the size, which must be a message's and within the
        // bound, else the call fails as for a malformed message (and the message counts as
        // empty). Every block of the message reads it alike.
        uint64_t T = 0;
        size_ok = stream_tokens(a.dev_bytes[w], 0, &T) && T <= d.T;
        d.T = size_ok ? T : 0;
        d.runs_off = 32 + 4 * d.T;
    }
    const uint64_t lc = c - d.chunk_base;
    // the call's control word starts clear: the first launch clears it, and every mark comes
    // from the second launch or the kernels after it
    if (kPass == 0 && c == 0 && threadIdx.x == 0) a.ctl->any_bad = 0u;
    if (lc == 0) {
        if (kPass == 0) {
            // (with more than kMax messages and sizes in device memory, the other chunks of the
            // message may read this entry as it changes: they take only fields that stay the
            // same, and T from the size themselves)
            if (threadIdx.x == 0 && (a.W <= kMax || a.dev_bytes)) a.tab[w] = d;
            if (d.T == 0)  // no token: its first token in every tile is 0 (= T)
                for (uint64_t tt = threadIdx.x; tt <= a.ntiles; tt += kPosThreads)
                    a.ts[tt * a.W + w] = 0;
        } else if (d.T == 0) {
            // the header of a message without tokens, checked once the first launch is done
            grid_dep_wait();
            if (threadIdx.x == 0 && (!size_ok || !header_ok(a, d))) mark_bad(a);
        }
        if (d.T == 0) return;
    } else if (lc * kDecChunk >= d.T) {
        // with sizes in device memory the chunks are laid out for each message's bound on T: the
        // chunks past its real end have nothing to do (and no later chunk of it looks back to
        // them)
        return;
    }
    constexpr int kPer = kDecChunk / kPosThreads;
    static_assert(kPer % 4 == 0 && kPer <= 32, "pairs of advances per word, one escape bit each");
    // this thread's tokens [j0, j0 + cnt) of the message
    const uint64_t j0 = lc * kDecChunk + (uint64_t)threadIdx.x * kPer;
    const uint32_t cnt = (uint32_t)(j0 >= d.T ? 0 : umin64(kPer, d.T - j0));
    // each token's advance (an escape skips 65535, another token run + 1 <= 65535) in 16 bits,
    // two per word, and which tokens are escapes
    uint32_t adv2[kPer / 2];
    uint32_t esc = 0, mine = 0;
    const uint8_t* runs_b = d.ptr + d.runs_off;
    if (!a.qbits && cnt == kPer) {
        // binary32 messages keep their runs block on a 4-byte boundary and pad the message to a
        // multiple of 4 bytes: the runs come two per 32-bit load
        const uint32_t* r2 = reinterpret_cast<const uint32_t*>(runs_b) + j0 / 2;
        uint32_t raw[kPer / 2];
#pragma unroll
        for (int k = 0; k < kPer / 2; ++k) raw[k] = r2[k];
#pragma unroll
        for (int k = 0; k < kPer / 2; ++k) {
            const uint32_t r0 = raw[k] & 0xFFFFu, r1 = raw[k] >> 16;
            const uint32_t a0 = (r0 == kRunEscape) ? kRunEscape : r0 + 1;
            const uint32_t a1 = (r1 == kRunEscape) ? kRunEscape : r1 + 1;
            esc |= (uint32_t)(r0 == kRunEscape) << (2 * k);
            esc |= (uint32_t)(r1 == kRunEscape) << (2 * k + 1);
            adv2[k] = a0 | (a1 << 16);
            mine += a0 + a1;
        }
    } else {
        const uint16_t* runs = reinterpret_cast<const uint16_t*>(runs_b);
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            uint32_t adv = 0;
            if ((uint32_t)i < cnt) {
                const uint32_t r = runs[j0 + i];
                adv = (r == kRunEscape) ? kRunEscape : r + 1;
                esc |= (uint32_t)(r == kRunEscape) << i;
            }
            if (i & 1) adv2[i / 2] |= adv << 16;
            else adv2[i / 2] = adv;
            mine += adv;
        }
    }
    uint32_t agg;
    const uint32_t ex = block_excl_scan<kPosThreads>(mine, s_scan, &agg);
    if (kPass == 0) {
        // the chunk's advances, published for the position pass (a message's first chunk: its
        // inclusive prefix); the header
        if (threadIdx.x == 0) st_relaxed(&a.st[c], (lc == 0 ? kFlagInc : kFlagAgg) | agg);
        return;
    }
    // the second launch: the first one's words, and the control word it cleared, from here on
    grid_dep_wait();
    if (lc == 0 && threadIdx.x == 0 && (!size_ok || !header_ok(a, d))) mark_bad(a);
    // a message's first chunk starts at end 0; the others look back over their predecessors,
    // whose words the aggregate pass has all written (kPosThreads of them per round trip)
    uint64_t base = 0;
    if (lc > 0)
        base = block_lookback<kPosThreads>(a.st, (uint32_t)c, agg, a.spin_limit, a.status, nullptr,
                                           s_lb32, s_lb64, false);
    if (cnt == 0) return;
    const uint64_t start = base + ex;  // the end of the token before this thread's first
    // ends up to lim (<= n) are positions inside the dense array
    const uint32_t lim = (start >= a.n) ? 0u : (uint32_t)umin64(a.n - start, 0xFFFFFFFFull);
    const uint32_t s32 = (uint32_t)start;  // exact while start < n
    uint32_t pos[kPer];
    uint32_t cum = 0;  // advances of this thread's tokens so far
    bool bad = false;
    const int32_t ntiles = (int32_t)a.ntiles;
    uint32_t* ts_w = a.ts + w;  // ts[t * W + w]
    // the tile of the previous token's position (-1 before a message's first token): the tiles
    // after it, up to this token's, have this token as their first
    int32_t qp = (start == 0) ? -1 : (int32_t)((s32 - 1u) / kDecTile);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        pos[i] = 0;
        if ((uint32_t)i >= cnt || bad) continue;
        const uint32_t adv = (i & 1) ? (adv2[i / 2] >> 16) : (adv2[i / 2] & 0xFFFFu);
        cum += adv;
        if (cum > lim) {  // past the end of the dense array: a malformed message
            bad = true;
            continue;
        }
        const uint32_t p = s32 + cum - 1u;  // this token's position
        pos[i] = ((esc >> i) & 1u) ? kEscPos : p;
        const int32_t q = (int32_t)(p / kDecTile);
        if (q != qp) {
            for (int32_t t = qp + 1; t <= min(q, ntiles); ++t)
                ts_w[(uint64_t)t * a.W] = (uint32_t)(j0 + i);
            qp = q;
        }
    }
    // the message's last token: every later tile has no token of it (its first is T)
    if (!bad && j0 + cnt == d.T)
        for (int32_t t = qp + 1; t <= ntiles; ++t) ts_w[(uint64_t)t * a.W] = (uint32_t)d.T;
    if (bad) {
        mark_bad(a);
        return;
    }
    // the positions: four 16-byte stores when the thread's 16 tokens are whole (message bases
    // in the position array are multiples of 4)
    uint32_t* out = a.pos + d.tok_base + j0;
    if (cnt == kPer) {
#pragma unroll
        for (int k = 0; k < kPer / 4; ++k)
            reinterpret_cast<uint4*>(out)[k] =
                make_uint4(pos[4 * k], pos[4 * k + 1], pos[4 * k + 2], pos[4 * k + 3]);
    } else {
#pragma unroll
        for (int i = 0; i < kPer; ++i)
            if ((uint32_t)i < cnt) out[i] = pos[i];
    }
}

// A message's tokens in rows [r0, r1) of the first-token table: [*first, *first + count).
// The table rises from 0 to T down each message's column; an entry that does not is reported as
// a corrupt call and read as no token, so a token index never leaves the message.
__device__ __forceinline__ uint32_t table_range(const DecArgs& a, uint64_t r0, uint64_t r1,
                                                int w, uint64_t T, uint32_t* first) {
    const uint32_t j0 = a.ts[r0 * a.W + w], j1 = a.ts[r1 * a.W + w];
    if (j0 > j1 || j1 > T) {
        report(a.status, DGC_ECORRUPT);
        *first = 0;
        return 0;
    }
    *first = j0;
    return j1 - j0;
}

// token j's value: binary32 bits (version 1) or the integer, sign-extended (version 2)
__device__ __forceinline__ uint32_t dec_value(const DecArgs& a, const DecStream& d, uint64_t j) {
    if (a.qbits == 8) return (uint32_t)(int32_t)reinterpret_cast<const int8_t*>(d.ptr + 32)[j];
    if (a.qbits == 16) return (uint32_t)(int32_t)reinterpret_cast<const int16_t*>(d.ptr + 32)[j];
    return reinterpret_cast<const uint32_t*>(d.ptr + 32)[j];
}

// an integer sum back to a value: one conversion, one division by the shared alpha
__device__ __forceinline__ float dequant(int32_t S, float alpha) {
    return __fdiv_rn(__int2float_rn(S), alpha);
}

// kInt: version-2 messages. Their integers are summed exactly (any order gives the same sum) and
// turned into a value once per position; a flag per entry records whether any message landed.
//
// Binary32 sums keep the learners' order at every position. A message's positions are
// distinct, so only tokens of different messages can meet at one position. The tile's tokens
// are staged (message-major, up to kDecCap at a time) and added in rounds: each round, every
// position still owed a value finds the smallest message index among its remaining tokens
// (a shared atomicMin) and that token alone adds itself, then clears the position's minimum for
// the next round. Positions that one message reaches finish in the first round; a round adds at
// most one value per position, so the number of rounds is the most tokens that meet at one
// position. Staged chunks follow each other in message order, so chunk boundaries keep the
// order too.
constexpr uint32_t kNoPos = 0xFFFFFFFFu;
template <bool kInt>
__global__ void __launch_bounds__(kThreads, 5) k_dec_tiles(DecArgs a) {
    constexpr int kPerThread = kDecCap / kThreads;  // staged tokens per thread
    static_assert(kPerThread * kThreads == kDecCap && kPerThread <= 32, "staging layout");
    __shared__ __align__(16) uint32_t s_accw[kDecTile];  // binary32 sums, or int32 sums
    __shared__ uint8_t s_touch[kInt ? kDecTile : 1];
    __shared__ __align__(16) uint32_t s_minw[kInt ? 1 : kDecTile];  // smallest message left
    __shared__ uint32_t s_pos[kDecCap];  // tile-local position, or kNoPos
    __shared__ uint32_t s_val[kDecCap];
    __shared__ uint32_t s_msg[kInt ? 1 : kDecCap];  // message index within the group
    __shared__ uint32_t s_off[kThreads + 1];
    __shared__ uint32_t s_first[kThreads];
    __shared__ uint64_t s_scan[33];
    __shared__ uint32_t s_fill;  // staging slots claimed by the warps (one-pass path)
    float* s_acc = reinterpret_cast<float*>(s_accw);
    int32_t* s_acci = reinterpret_cast<int32_t*>(s_accw);
    grid_dep_wait();
    if (ld_relaxed_u32(&a.ctl->any_bad)) return;  // a malformed message: leave dense as it is
    const uint64_t t = blockIdx.x;
    const uint64_t p0 = t * kDecTile;
    const uint32_t len = (uint32_t)umin64(kDecTile, a.n - p0);
    const bool vec = (len == kDecTile) && ((reinterpret_cast<uintptr_t>(a.dense) & 15u) == 0);
    const bool load = !kInt && a.accumulate && !a.apply;  // apply mode sums from +0
    if (kInt) {
        for (uint32_t i = threadIdx.x; i < kDecTile; i += kThreads) {
            s_acci[i] = 0;
            s_touch[i] = 0;
        }
    } else {
        for (uint32_t i = threadIdx.x; i < kDecTile / 4; i += kThreads)
            reinterpret_cast<uint4*>(s_minw)[i] = make_uint4(kNoPos, kNoPos, kNoPos, kNoPos);
        if (vec && load) {
            for (uint32_t i = threadIdx.x; i < kDecTile / 4; i += kThreads)
                reinterpret_cast<float4*>(s_acc)[i] = reinterpret_cast<const float4*>(a.dense + p0)[i];
        } else if (vec) {
            for (uint32_t i = threadIdx.x; i < kDecTile / 4; i += kThreads)
                reinterpret_cast<float4*>(s_acc)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            for (uint32_t i = threadIdx.x; i < kDecTile; i += kThreads)
                s_acc[i] = (load && i < len) ? a.dense[p0 + i] : 0.0f;
        }
    }
    if (threadIdx.x == 0) s_fill = 0;
    __syncthreads();  // the cleared tile, s_minw and s_fill before any staging
    // the staged tokens this thread owns in the rounds: slots tid + k kThreads
    auto rounds = [&](uint32_t m) {
        uint32_t act = 0;
#pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            const uint32_t i = threadIdx.x + (uint32_t)k * kThreads;
            if (i < m && s_pos[i] != kNoPos) act |= 1u << k;
        }
        // every position still owed a value takes the token of its smallest message; a
        // barrier closes each round (s_minw is kNoPos everywhere between rounds)
        do {
#pragma unroll
            for (int k = 0; k < kPerThread; ++k) {
                const uint32_t i = threadIdx.x + (uint32_t)k * kThreads;
                if (act & (1u << k)) atomicMin(&s_minw[s_pos[i]], s_msg[i]);
            }
            __syncthreads();
#pragma unroll
            for (int k = 0; k < kPerThread; ++k) {
                const uint32_t i = threadIdx.x + (uint32_t)k * kThreads;
                if (!(act & (1u << k))) continue;
                const uint32_t lp = s_pos[i];
                // the one token of the smallest message left at lp (another token there
                // may already see the cleared word: it never equals a message index)
                if (s_minw[lp] == s_msg[i]) {
                    s_acc[lp] = __fadd_rn(s_acc[lp], __uint_as_float(s_val[i]));
                    s_minw[lp] = kNoPos;
                    act &= ~(1u << k);
                }
            }
        } while (__syncthreads_or(act != 0));
    };
    // Up to kThreads messages: thread w owns message w. It reads the message's first and end
    // token in this tile from the table; a warp scan places the warp's tokens, one shared atomic
    // per warp claims a region of the staging slots, and every thread stages its own message's
    // tokens there (integer messages are added at once: their sum does not depend on order). The
    // order of the regions does not matter, since a round adds by message index. When the tile's
    // tokens do not fit the staging slots, the chunked path below stages them message-major.
    bool done = false;
    if (a.W <= kThreads) {
        const int w = threadIdx.x;
        uint32_t cnt = 0, first = 0;
        if (w < a.W && a.tab[w].T > 0) {
            cnt = table_range(a, t, t + 1, w, a.tab[w].T, &first);
        }
        const int lane = threadIdx.x & 31;
        const uint32_t incl = warp_incl_scan(cnt);
        const uint32_t wtot = __shfl_sync(0xFFFFFFFFu, incl, 31);
        uint32_t base = 0;
        if (lane == 31 && !kInt && wtot) base = atomicAdd(&s_fill, wtot);
        base = __shfl_sync(0xFFFFFFFFu, base, 31);
        const bool fits = kInt || base + wtot <= (uint32_t)kDecCap;
        if (cnt > 0 && fits) {
            const DecStream& d = a.tab[w];
            const uint32_t at = base + incl - cnt;
            auto stage = [&](uint32_t q, uint32_t p, uint32_t raw) {
                const bool in = p != kEscPos && p >= p0 && p < p0 + len;
                if (kInt) {
                    if (in) {
                        atomicAdd(&s_acci[p - p0], (int32_t)raw);
                        s_touch[p - p0] = 1;
                    }
                } else {
                    s_pos[at + q] = in ? (uint32_t)(p - p0) : kNoPos;
                    s_val[at + q] = raw;
                    s_msg[at + q] = (uint32_t)w;
                }
            };
            constexpr uint32_t kBatch = 8;  // loads in flight before any is used
            uint32_t pb[kBatch], rb[kBatch];
#pragma unroll
            for (uint32_t q = 0; q < kBatch; ++q)
                if (q < cnt) {
                    pb[q] = a.pos[d.tok_base + first + q];
                    rb[q] = dec_value(a, d, (uint64_t)first + q);
                }
#pragma unroll
            for (uint32_t q = 0; q < kBatch; ++q)
                if (q < cnt) stage(q, pb[q], rb[q]);
            for (uint32_t q = kBatch; q < cnt; ++q) {
                const uint64_t j = (uint64_t)first + q;
                stage(q, a.pos[d.tok_base + j], dec_value(a, d, j));
            }
        }
        const bool overflow = __syncthreads_or(!fits);
        if (!overflow) {
            if (!kInt && s_fill > 0) rounds(s_fill);
            done = true;
        }
    }
    for (int wb = 0; !done && wb < a.W; wb += kThreads) {
        const int w = wb + threadIdx.x;
        uint32_t cnt = 0, first = 0;
        if (w < a.W && a.tab[w].T > 0) {
            cnt = table_range(a, t, t + 1, w, a.tab[w].T, &first);
        }
        uint64_t total;
        const uint64_t ex = block_excl_scan<kThreads>((uint64_t)cnt, s_scan, &total);
        s_off[threadIdx.x] = (uint32_t)ex;
        s_first[threadIdx.x] = first;
        if (threadIdx.x == 0) s_off[kThreads] = (uint32_t)total;
        __syncthreads();
        const int nw = min(kThreads, a.W - wb);
        if (total <= kDecCap) {
            // one chunk (the common case): each message's own thread stages its few tokens at
            // the message's offset, so no token searches for its message
            if (threadIdx.x < nw && cnt > 0) {
                const DecStream& d = a.tab[wb + threadIdx.x];
                const uint32_t at = (uint32_t)ex;
                auto stage = [&](uint32_t q, uint32_t p, uint32_t raw) {
                    const bool in = p != kEscPos && p >= p0 && p < p0 + len;
                    if (kInt) {
                        if (in) {
                            atomicAdd(&s_acci[p - p0], (int32_t)raw);
                            s_touch[p - p0] = 1;
                        }
                    } else {
                        s_pos[at + q] = in ? (uint32_t)(p - p0) : kNoPos;
                        s_val[at + q] = raw;
                        s_msg[at + q] = (uint32_t)threadIdx.x;
                    }
                };
                // the first kBatch tokens' loads all in flight before any is used
                constexpr uint32_t kBatch = 8;
                uint32_t pb[kBatch], rb[kBatch];
#pragma unroll
                for (uint32_t q = 0; q < kBatch; ++q)
                    if (q < cnt) {
                        pb[q] = a.pos[d.tok_base + first + q];
                        rb[q] = dec_value(a, d, (uint64_t)first + q);
                    }
#pragma unroll
                for (uint32_t q = 0; q < kBatch; ++q)
                    if (q < cnt) stage(q, pb[q], rb[q]);
                for (uint32_t q = kBatch; q < cnt; ++q) {
                    const uint64_t j = (uint64_t)first + q;
                    stage(q, a.pos[d.tok_base + j], dec_value(a, d, j));
                }
            }
            __syncthreads();
            if (!kInt && total > 0) rounds((uint32_t)total);
            continue;
        }
        for (uint32_t r0 = 0; r0 < total; r0 += kDecCap) {
            const uint32_t m = (uint32_t)umin64(kDecCap, total - r0);
#pragma unroll
            for (int k = 0; k < kPerThread; ++k) {
                const uint32_t i = threadIdx.x + (uint32_t)k * kThreads;
                if (i >= m) break;
                const uint32_t f = r0 + i;
                int l = 0, h = nw;  // message of flattened token f
                while (h - l > 1) {
                    const int mid = (l + h) >> 1;
                    if (s_off[mid] <= f) l = mid; else h = mid;
                }
                const DecStream& d = a.tab[wb + l];
                const uint64_t j = s_first[l] + (f - s_off[l]);
                const uint32_t p = a.pos[d.tok_base + j];
                const uint32_t raw = dec_value(a, d, j);
                const bool in = p != kEscPos && p >= p0 && p < p0 + len;
                if (kInt) {
                    if (in) {
                        atomicAdd(&s_acci[p - p0], (int32_t)raw);
                        s_touch[p - p0] = 1;
                    }
                } else {
                    s_pos[i] = in ? (uint32_t)(p - p0) : kNoPos;
                    s_val[i] = raw;
                    s_msg[i] = (uint32_t)l;
                }
            }
            if (!kInt) rounds(m);  // each thread reads back only slots it staged itself
            else __syncthreads();  // the staged chunk is consumed before the next one is staged
        }
    }
    __syncthreads();
    // Modes that read the output first (the SGD step, accumulation of integer sums) load every
    // value this thread needs before any arithmetic, so a tile costs one round trip to memory
    // instead of one per entry; only the entries that change are written.
    constexpr int kOut = kDecTile / kThreads;
    if (kInt) {
        if (a.apply || a.accumulate) {
            float o[kOut];
#pragma unroll
            for (int k = 0; k < kOut; ++k) {
                const uint32_t i = threadIdx.x + (uint32_t)k * kThreads;
                const bool need = i < len && (a.apply ? s_acci[i] != 0 : s_touch[i] != 0);
                o[k] = need ? a.dense[p0 + i] : 0.0f;
            }
#pragma unroll
            for (int k = 0; k < kOut; ++k) {
                const uint32_t i = threadIdx.x + (uint32_t)k * kThreads;
                if (i >= len) break;
                const int32_t S = s_acci[i];
                if (a.apply) {  // S == 0: the step is the identity
                    if (S) a.dense[p0 + i] = __fmaf_rn(a.neg_lr, dequant(S, a.alpha), o[k]);
                } else if (s_touch[i]) {  // one addition where a message landed
                    a.dense[p0 + i] = __fadd_rn(o[k], dequant(S, a.alpha));
                }
            }
        } else {
            for (uint32_t i = threadIdx.x; i < len; i += kThreads)
                a.dense[p0 + i] = dequant(s_acci[i], a.alpha);
        }
    } else if (a.apply) {
        // a sum that starts at +0 is +0 wherever no message lands (x + y is -0 only for two -0
        // addends), and fma(neg_lr, +0, w) == w for a finite neg_lr with its sign bit set: those
        // entries are left alone, the others take the step
        float o[kOut];
#pragma unroll
        for (int k = 0; k < kOut; ++k) {
            const uint32_t i = threadIdx.x + (uint32_t)k * kThreads;
            o[k] = (i < len && __float_as_uint(s_acc[i]) != 0u) ? a.dense[p0 + i] : 0.0f;
        }
#pragma unroll
        for (int k = 0; k < kOut; ++k) {
            const uint32_t i = threadIdx.x + (uint32_t)k * kThreads;
            if (i >= len) break;
            const float t = s_acc[i];
            if (__float_as_uint(t) != 0u) a.dense[p0 + i] = __fmaf_rn(a.neg_lr, t, o[k]);
        }
    } else if (vec) {
        for (uint32_t i = threadIdx.x; i < kDecTile / 4; i += kThreads)
            reinterpret_cast<float4*>(a.dense + p0)[i] = reinterpret_cast<const float4*>(s_acc)[i];
    } else {
        for (uint32_t i = threadIdx.x; i < len; i += kThreads) a.dense[p0 + i] = s_acc[i];
    }
}

// Binary32 sums of several messages into the dense array (not the SGD step, not integer
// messages), one tile of kSumTile entries (kSumTile / kDecTile rows of the first-token table)
// per block of kSumThreads threads. The block first stores +0 over its tile (unless
// accumulating). The tile's tokens are staged in shared memory, kSumCap at a time, message-major
// and spread over all threads, so neighbouring threads load neighbouring tokens of a message.
// Staging marks each position in two bitmaps: one token landed, a second one landed. After a
// barrier, a token whose position holds no other adds its value onto the position's value (+0
// in the first round of a plain sum, the stored value otherwise) and stores it; the rest, where
// several messages meet, go to a short list, and there the token of the smallest message adds
// the position's values in message order. A message reaches a position at most once, so the
// smallest message is unique. Messages go in groups of kSumThreads, and a group whose tokens
// exceed the staging slots goes in message-major rounds; groups and rounds follow the message
// order and every round adds onto what the earlier ones stored, so each position's sum takes the
// learners' order throughout.
constexpr int kSumTile = 4 * kDecTile;
constexpr int kSumRows = kSumTile / kDecTile;  // first-token table rows per tile
constexpr int kSumThreads = 256;
constexpr int kSumCap = 2048;  // tokens staged per round
constexpr int kSumWords = kSumTile / 32;
// Order this thread's completed bulk-copy (async-proxy) writes to global memory before its later
// generic-proxy accesses, so that a barrier after it orders them for the whole block.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

constexpr uint16_t kNoLp = 0xFFFFu;  // an escape, or a position outside the tile
static_assert(kSumCap <= 0xFFFF && kSumTile < 0xFFFF, "16-bit slots and positions");

__global__ void __launch_bounds__(kSumThreads, 5) k_dec_sum(DecArgs a) {
    constexpr int kPer = kSumCap / kSumThreads;  // staged slots per thread
    __shared__ uint32_t s_val[kSumCap];
    __shared__ uint16_t s_lp[kSumCap];     // position within the tile, or kNoLp
    __shared__ uint16_t s_msg[kSumCap];    // message index within the group
    __shared__ uint16_t s_multi[kSumCap];  // slots whose position holds several tokens
    __shared__ uint16_t s_sorted[kSumCap]; // the same slots by (position, message)
    __shared__ uint32_t s_key[kSumCap];    // their (position, message), in s_multi's order
    __shared__ uint32_t s_one[kSumWords];  // a token landed at the position
    __shared__ uint32_t s_two[kSumWords];  // a second token landed there
    __shared__ uint64_t s_tb[kSumThreads];          // the group's messages: position base
    __shared__ const uint8_t* s_vp[kSumThreads];    // and their values
    __shared__ uint32_t s_scan[33];
    __shared__ uint32_t s_nmulti;
    __shared__ __align__(128) float s_zero[1024];  // the source of the tile's zeros
    grid_dep_wait();
    if (ld_relaxed_u32(&a.ctl->any_bad)) return;  // a malformed message: leave dense as it is
    const uint64_t p0 = (uint64_t)blockIdx.x * kSumTile;
    const uint32_t len = (uint32_t)umin64(kSumTile, a.n - p0);
    const uint64_t row0 = (uint64_t)blockIdx.x * kSumRows;
    const uint64_t row1 = umin64(row0 + kSumRows, a.ntiles);
    float* out = a.dense + p0;
    // the plain sum starts from +0 everywhere: the tile is cleared once, before the barrier that
    // precedes every store of a sum
    bool cleared = a.accumulate != 0;
    // a whole, aligned tile of a plain sum: its zeros go out as 16 bulk copies of a zeroed 4 KB
    // shared buffer, issued by one thread at once; that thread waits for them (and fences them
    // from the generic stores) before the barrier that precedes the first stored sum
    const bool bulk = !cleared && len == kSumTile && (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
    if (bulk) {
        for (uint32_t i = threadIdx.x; i < 1024; i += kSumThreads) s_zero[i] = 0.0f;
        fence_proxy_async_smem();
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int c = 0; c < kSumTile / 1024; ++c) bulk_s2g(out + c * 1024, s_zero, 4096u);
            bulk_commit();
        }
        cleared = true;
    }
    bool waited = false;  // (the same in every thread)
    auto bulk_done = [&]() {
        if (bulk && !waited && threadIdx.x == 0) {
            bulk_wait_all();
            fence_proxy_async_global();
        }
        waited = true;
    };
    // otherwise (a partial or unaligned tile) plain stores, issued once the first round's loads
    // are in flight (they would wait behind the stores otherwise)
    auto clear_tile = [&]() {
        if (len == kSumTile && (reinterpret_cast<uintptr_t>(out) & 15u) == 0) {
#pragma unroll 4
            for (uint32_t i = threadIdx.x; i < kSumTile / 4; i += kSumThreads)
                reinterpret_cast<float4*>(out)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            for (uint32_t i = threadIdx.x; i < len; i += kSumThreads) out[i] = 0.0f;
        }
        cleared = true;
    };
    auto clear_marks = [&]() {
        for (uint32_t i = threadIdx.x; i < kSumWords; i += kSumThreads) {
            s_one[i] = 0;
            s_two[i] = 0;
        }
        if (threadIdx.x == 0) s_nmulti = 0;
    };
    clear_marks();
    bool first = !a.accumulate;  // no round has stored a sum yet: they start from +0
    for (int wb = 0; wb < a.W; wb += kSumThreads) {
        const int w = wb + (int)threadIdx.x;
        uint32_t cnt = 0, j0 = 0;
        // (the position kernel writes every message's column, an empty message's too)
        if (w < a.W) cnt = table_range(a, row0, row1, w, a.tab[w].T, &j0);
        if (w < a.W) {  // where the message's positions and values start
            const DecStream& d = a.tab[w];
            s_tb[threadIdx.x] = d.tok_base;
            s_vp[threadIdx.x] = d.ptr + 32;
        }
        uint32_t total;
        const uint32_t ex = block_excl_scan<kSumThreads>(cnt, s_scan, &total);
        const int nw = min(kSumThreads, a.W - wb);
        for (uint32_t r0 = 0; r0 < total; r0 += kSumCap) {
            const uint32_t m = min((uint32_t)kSumCap, total - r0);
            // stage in two steps: each message's own thread writes, for its tokens among this
            // round's, the message and the token's index into their slots; then every thread
            // loads the position and value of its slots (neighbouring slots, neighbouring tokens
            // of one message), all of its loads issued before any is used
            if ((int)threadIdx.x < nw && ex < r0 + m && ex + cnt > r0) {
                const uint32_t f0 = max(ex, r0), f1 = min(ex + cnt, r0 + m);  // flattened
                for (uint32_t f = f0; f < f1; ++f) {
                    s_val[f - r0] = j0 + (f - ex);
                    s_msg[f - r0] = (uint16_t)threadIdx.x;
                }
            }
            __syncthreads();  // the round's slots name their tokens
            uint32_t pv[kPer], rv[kPer];
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const uint32_t i = threadIdx.x + (uint32_t)k * kSumThreads;
                if (i >= m) continue;
                const uint32_t l = s_msg[i], j = s_val[i];
                pv[k] = a.pos[s_tb[l] + j];
                // binary32 bits, or (one integer message) the integer, sign-extended
                const uint8_t* vb = s_vp[l];
                rv[k] = a.qbits == 8    ? (uint32_t)(int32_t)reinterpret_cast<const int8_t*>(vb)[j]
                        : a.qbits == 16 ? (uint32_t)(int32_t)reinterpret_cast<const int16_t*>(vb)[j]
                                        : reinterpret_cast<const uint32_t*>(vb)[j];
            }
            if (!cleared) clear_tile();
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const uint32_t i = threadIdx.x + (uint32_t)k * kSumThreads;
                if (i >= m) continue;
                const uint32_t p = pv[k];
                const bool in = p != kEscPos && p >= p0 && p < p0 + len;
                const uint32_t lp = in ? (uint32_t)(p - p0) : kNoLp;
                s_lp[i] = (uint16_t)lp;
                s_val[i] = rv[k];
                if (in) {
                    const uint32_t bit = 1u << (lp & 31);
                    if (atomicOr(&s_one[lp >> 5], bit) & bit) atomicOr(&s_two[lp >> 5], bit);
                }
            }
            bulk_done();
            __syncthreads();  // the round's tokens and marks
            // a position with one token of the round: that token's value, added on
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const uint32_t i = threadIdx.x + (uint32_t)k * kSumThreads;
                if (i >= m) continue;
                const uint32_t lp = s_lp[i];
                if (lp == kNoLp) continue;
                if (s_two[lp >> 5] & (1u << (lp & 31))) {
                    const uint32_t at = atomicAdd(&s_nmulti, 1u);
                    s_multi[at] = (uint16_t)i;
                    s_key[at] = (lp << 16) | s_msg[i];
                    continue;
                }
                if (a.qbits) {  // one message of integers: one dequantization, added on
                    const float x = dequant((int32_t)s_val[i], a.alpha);
                    out[lp] = a.accumulate ? __fadd_rn(out[lp], x) : x;
                } else {
                    out[lp] = __fadd_rn(first ? 0.0f : out[lp], __uint_as_float(s_val[i]));
                }
            }
            __syncthreads();  // the list of tokens at shared positions
            // positions several messages reach: those tokens sorted by (position, message), each
            // by its rank among them; then the first token of each position adds the position's
            // values in message order
            const uint32_t nm = s_nmulti;
            if (nm > 0) {  // block-uniform
                for (uint32_t k = threadIdx.x; k < nm; k += kSumThreads) {
                    const uint32_t key = s_key[k];
                    uint32_t rank = 0;
                    for (uint32_t q = 0; q < nm; ++q) rank += s_key[q] < key;
                    s_sorted[rank] = s_multi[k];  // keys are distinct: ranks are too
                }
                __syncthreads();
                for (uint32_t r = threadIdx.x; r < nm; r += kSumThreads) {
                    const uint32_t i = s_sorted[r];
                    const uint32_t lp = s_lp[i];
                    if (r > 0 && s_lp[s_sorted[r - 1]] == lp) continue;
                    float acc = __fadd_rn(first ? 0.0f : out[lp], __uint_as_float(s_val[i]));
                    for (uint32_t r2 = r + 1; r2 < nm; ++r2) {
                        const uint32_t i2 = s_sorted[r2];
                        if (s_lp[i2] != lp) break;
                        acc = __fadd_rn(acc, __uint_as_float(s_val[i2]));
                    }
                    out[lp] = acc;
                }
            }
            first = false;
            if (r0 + kSumCap < total || wb + kSumThreads < a.W) {
                // another round follows: its staging waits for every use of this one, and its
                // marks start clear (the stored sums are visible to it after the barriers)
                __syncthreads();
                clear_marks();
                __syncthreads();
            }
        }
    }
    if (!cleared) clear_tile();  // a tile no token reaches
    bulk_done();  // (the zeros must be out before the block ends, even with no token)
}

// The SGD step from one message (W = 1): its positions are distinct, so each value token takes
// the step at its own position (the one-message sum there is +0 + x).
__global__ void __launch_bounds__(kThreads) k_dec_scatter1(DecArgs a) {
    grid_dep_wait();
    if (ld_relaxed_u32(&a.ctl->any_bad)) return;  // a malformed message: leave dense as it is
    const DecStream d = a.tab[0];
    const uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= d.T) return;
    const uint32_t p = a.pos[d.tok_base + j];
    if (p == kEscPos || p >= a.n) return;
    const uint32_t raw = dec_value(a, d, j);
    const float x = a.qbits ? dequant((int32_t)raw, a.alpha) : __uint_as_float(raw);
    a.dense[p] = __fmaf_rn(a.neg_lr, __fadd_rn(0.0f, x), a.dense[p]);
}

// ---------------------------------------------------------------- shared-set sums
// out[j] = ((+0 + vals[0][j]) + vals[1][j]) + ... : the learners in order, as the decoders add
// them. Consecutive threads read consecutive entries of each learner's vector.
__global__ void __launch_bounds__(kThreads) k_sum_shared(const float* const* vals, int32_t W,
                                                        const int64_t* count, uint64_t max_count,
                                                        float* out, int32_t* status) {
    const int64_t c = *count;
    if (c < 0 || (uint64_t)c > max_count) {
        if (blockIdx.x == 0 && threadIdx.x == 0) report(status, DGC_EINVAL);
        return;
    }
    for (uint64_t j = (uint64_t)blockIdx.x * kThreads + threadIdx.x; j < (uint64_t)c;
         j += (uint64_t)gridDim.x * kThreads) {
        float acc = 0.0f;
        for (int32_t w = 0; w < W; ++w) acc = __fadd_rn(acc, vals[w][j]);
        out[j] = acc;
    }
}

// A launch that may overlap the end of the kernel ahead of it in the stream (the kernel waits
// for it with grid_dep_wait before reading what it wrote).
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), uint64_t grid, unsigned block,
                             cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

struct DecLayout {
    size_t ctl, tab, pos, st, ts, total;
    uint64_t sum_T, pos_len, nchunks, ntiles;
};

// bounds: stream_bytes are upper bounds on binary32 messages' sizes (their T found on the
// device); else the sizes themselves
int dec_layout(int32_t W, const uint64_t* stream_bytes, int64_t n, int qbits, DecLayout* L,
               std::vector<DecStream>* tab, bool bounds = false) {
    L->sum_T = 0;
    L->pos_len = 0;
    L->nchunks = 0;
    for (int w = 0; w < W; ++w) {
        uint64_t T;
        if (bounds) T = stream_bytes[w] >= 32 ? (stream_bytes[w] - 32) / 6 : 0;
        else if (!stream_tokens(stream_bytes[w], qbits, &T)) return DGC_ECORRUPT;
        const uint64_t ro = qbits ? q_runs_offset(T, qbits) : 32 + 4 * T;
        // a message's positions start on a multiple of 4 entries (16-byte stores)
        if (tab) (*tab)[w] = DecStream{nullptr, T, L->pos_len, L->nchunks, ro};
        L->sum_T += T;
        L->pos_len += (T + 3) & ~3ull;
        L->nchunks += std::max<uint64_t>(1, (T + kDecChunk - 1) / kDecChunk);  // one at least
    }
    if (tab) (*tab)[W] = DecStream{nullptr, 0, L->pos_len, L->nchunks, 0};
    L->ntiles = ((uint64_t)n + kDecTile - 1) / kDecTile;
    size_t o = 0;
    auto take = [&](size_t b) { size_t at = o; o = align256(o + b); return at; };
    L->ctl = take(sizeof(DecCtl));
    L->st = take(sizeof(uint64_t) * (size_t)(L->nchunks + 1));
    L->tab = take(sizeof(DecStream) * (size_t)(W + 1));
    L->pos = take(sizeof(uint32_t) * (size_t)L->pos_len);
    L->ts = take(sizeof(uint32_t) * (size_t)(L->ntiles + 1) * (size_t)(W > 0 ? W : 1));
    L->total = o;
    return DGC_OK;
}

}  // namespace
}  // namespace dgc

using namespace dgc;

extern "C" int dgc_encode_max_bytes(int64_t max_count, int64_t n, uint64_t* bytes) {
    if (!bytes || max_count < 0 || n < 0) return DGC_EINVAL;
    if (n > 0xFFFFFFFFll) return DGC_EUNSUPPORTED;
    const uint64_t T = (uint64_t)max_count + (uint64_t)n / kRunEscape;
    *bytes = 32 + 6 * T + 2;
    return DGC_OK;
}

extern "C" int dgc_encode_workspace(int64_t max_count, size_t* bytes) {
    if (!bytes || max_count < 0) return DGC_EINVAL;
    *bytes = align256(sizeof(EncCtl)) + align256(sizeof(uint64_t) * kEncBlocks);
    return DGC_OK;
}

namespace {
int encode_impl(const uint32_t* idx, const float* val, const int64_t* count, int64_t max_count,
                int64_t n, int32_t qbits, float alpha, float* v, uint8_t* out, uint64_t out_cap,
                uint64_t* out_bytes, int32_t* status, void* ws, size_t ws_bytes,
                dgc_stream_t stream) {
    if (max_count < 0 || n < 0) return DGC_EINVAL;
    if (n > 0xFFFFFFFFll || max_count > 0xFFFFFFFFll) return DGC_EUNSUPPORTED;
    if (!count || !out || !out_bytes || !status || !ws) return DGC_EINVAL;
    if (max_count > 0 && (!idx || !val)) return DGC_EINVAL;
    if (((uintptr_t)out & 15u) != 0 || ((uintptr_t)ws & 255u) != 0) return DGC_EINVAL;
    size_t need;
    dgc_encode_workspace(max_count, &need);
    if (ws_bytes < need) return DGC_EINVAL;
    EncArgs a{};
    a.idx = idx;
    a.val = val;
    a.count = count;
    a.max_count = (uint64_t)max_count;
    a.n = (uint64_t)n;
    a.out = out;
    a.out_cap = out_cap;
    a.out_bytes = out_bytes;
    a.status = status;
    a.qbits = qbits;
    a.alpha = alpha;
    a.v = v;
    char* w = static_cast<char*>(ws);
    a.ctl = reinterpret_cast<EncCtl*>(w);
    a.tot = reinterpret_cast<uint64_t*>(w + align256(sizeof(EncCtl)));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int sms = dgc_internal_sm_count();
    if (sms <= 0) return DGC_ECUDA;
    const int G = std::min(kEncBlocks, 2 * sms);
    // no memset: the scan kernel writes the control words; the count kernel is an ordinary
    // launch (it reads what came before the call), the other two may start while the one ahead
    // of them finishes
    k_enc_count<<<G, kThreads, 0, s>>>(a);
    const cudaError_t e1 = launch_dependent(k_enc_scan, 1, 1024, s, a, G);
    const cudaError_t e2 = launch_dependent(k_enc_write, (uint64_t)G, kThreads, s, a);
    dgc_internal_count_launches(3);
    if (e1 != cudaSuccess || e2 != cudaSuccess || cudaPeekAtLastError() != cudaSuccess) {
        cudaGetLastError();
        return DGC_ECUDA;
    }
    return DGC_OK;
}
}  // namespace

extern "C" int dgc_encode(const uint32_t* idx, const float* val, const int64_t* count,
                          int64_t max_count, int64_t n, uint8_t* out, uint64_t out_cap,
                          uint64_t* out_bytes, int32_t* status, void* ws, size_t ws_bytes,
                          dgc_stream_t stream) {
    return encode_impl(idx, val, count, max_count, n, 0, 0.0f, nullptr, out, out_cap, out_bytes,
                       status, ws, ws_bytes, stream);
}

extern "C" int dgc_encode_quant(const uint32_t* idx, const float* val, const int64_t* count,
                                int64_t max_count, int64_t n, float alpha, int32_t bits,
                                float* v, uint8_t* out, uint64_t out_cap, uint64_t* out_bytes,
                                int32_t* status, void* ws, size_t ws_bytes, dgc_stream_t stream) {
    if ((bits != 8 && bits != 16) || !std::isfinite(alpha) || !(alpha > 0.0f)) return DGC_EINVAL;
    return encode_impl(idx, val, count, max_count, n, bits, alpha, v, out, out_cap, out_bytes,
                       status, ws, ws_bytes, stream);
}

namespace {
int decode_workspace_impl(int32_t W, const uint64_t* stream_bytes, int64_t n, int32_t qbits,
                          size_t* bytes, bool bounds = false) {
    if (!bytes || W < 0 || n < 0 || (W > 0 && !stream_bytes)) return DGC_EINVAL;
    if (n > 0xFFFFFFFFll) return DGC_EUNSUPPORTED;
    DecLayout L;
    const int rc = dec_layout(W, stream_bytes, n, qbits, &L, nullptr, bounds);
    if (rc) return rc;
    *bytes = L.total;
    return DGC_OK;
}
}  // namespace

extern "C" int dgc_decode_workspace(int32_t W, const uint64_t* stream_bytes, int64_t n,
                                    size_t* bytes) {
    return decode_workspace_impl(W, stream_bytes, n, 0, bytes);
}

extern "C" int dgc_decode_workspace_bound(int32_t W, const uint64_t* max_bytes, int64_t n,
                                          size_t* bytes) {
    return decode_workspace_impl(W, max_bytes, n, 0, bytes, true);
}

extern "C" int dgc_decode_workspace_quant(int32_t W, const uint64_t* stream_bytes, int64_t n,
                                          int32_t bits, size_t* bytes) {
    if (bits != 8 && bits != 16) return DGC_EINVAL;
    return decode_workspace_impl(W, stream_bytes, n, bits, bytes);
}

namespace {
// dev_bytes: the message sizes in device memory (stream_bytes then holds host bounds on them)
int decode_impl(const uint8_t* const* streams, const uint64_t* stream_bytes, int32_t W,
                float* dense, int64_t n, int32_t accumulate, int32_t apply, float lr,
                int32_t qbits, float alpha, int32_t* status, void* ws, size_t ws_bytes,
                dgc_stream_t stream, const uint64_t* dev_bytes = nullptr) {
    if (W < 0 || n < 0) return DGC_EINVAL;
    if (n > 0xFFFFFFFFll) return DGC_EUNSUPPORTED;
    if (W > 0 && (!streams || !stream_bytes)) return DGC_EINVAL;
    if (!status || !ws || (n > 0 && !dense)) return DGC_EINVAL;
    if (((uintptr_t)ws & 255u) != 0) return DGC_EINVAL;
    for (int w = 0; w < W; ++w)
        if (!streams[w] || ((uintptr_t)streams[w] & 15u) != 0) return DGC_EINVAL;
    if (W > 0 && dev_bytes && ((uintptr_t)dev_bytes & 7u) != 0) return DGC_EINVAL;
    std::vector<DecStream> tab((size_t)W + 1);
    DecLayout L;
    int rc = dec_layout(W, stream_bytes, n, qbits, &L, &tab, dev_bytes != nullptr);
    if (rc) return rc;
    if (L.sum_T > 0xFFFFFFFFull) return DGC_EUNSUPPORTED;
    if (ws_bytes < L.total) return DGC_EINVAL;
    for (int w = 0; w < W; ++w) tab[w].ptr = streams[w];
    char* p = static_cast<char*>(ws);
    DecArgs a{};
    a.tab = reinterpret_cast<DecStream*>(p + L.tab);
    a.W = W;
    a.n = (uint64_t)n;
    a.dense = dense;
    a.accumulate = accumulate ? 1 : 0;
    a.apply = apply ? 1 : 0;
    a.neg_lr = -lr;
    a.qbits = qbits;
    a.alpha = alpha;
    a.status = status;
    a.ctl = reinterpret_cast<DecCtl*>(p + L.ctl);
    a.pos = reinterpret_cast<uint32_t*>(p + L.pos);
    a.st = reinterpret_cast<uint64_t*>(p + L.st);
    a.ts = reinterpret_cast<uint32_t*>(p + L.ts);
    a.dev_bytes = dev_bytes;
    a.ntiles = L.ntiles;
    a.nchunks = L.nchunks;
    a.spin_limit = kDefaultSpinLimit;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the table of messages goes with the first kernel's parameters when it is small; else by a
    // pageable copy (staged before this function returns, so the host vector may go away)
    if (W > kDecInline && cudaMemcpyAsync(p + L.tab, tab.data(), sizeof(DecStream) * tab.size(),
                                          cudaMemcpyHostToDevice, s) != cudaSuccess)
        return DGC_ECUDA;
    // the control word: cleared by the first position launch when there is one; the look-back
    // words need no clearing (the second launch reads only words the first wrote in this call)
    if (W == 0 && cudaMemsetAsync(p + L.ctl, 0, sizeof(DecCtl), s) != cudaSuccess)
        return DGC_ECUDA;
    // the first launch is ordinary (it reads what came before the call); every later one may
    // start while the one ahead of it finishes
    uint64_t launches = 0;
    cudaError_t e = cudaSuccess;
    auto ok = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
    if (W == 1) {  // the table of one message: a small launch
        DecTabInline<1> inl{};
        for (int w = 0; w <= W; ++w) inl.e[w] = tab[w];
        k_dec_pos<1, 0><<<(unsigned)L.nchunks, kPosThreads, 0, s>>>(a, inl);
        ok(launch_dependent(k_dec_pos<1, 1>, L.nchunks, kPosThreads, s, a, inl));
        launches += 2;
    } else if (W > 1) {
        DecTabInline<kDecInline> inl{};
        if (W <= kDecInline)
            for (int w = 0; w <= W; ++w) inl.e[w] = tab[w];
        k_dec_pos<kDecInline, 0><<<(unsigned)L.nchunks, kPosThreads, 0, s>>>(a, inl);
        ok(launch_dependent(k_dec_pos<kDecInline, 1>, L.nchunks, kPosThreads, s, a, inl));
        launches += 2;
    }
    const uint64_t sum_grid = (L.ntiles + kSumRows - 1) / kSumRows;
    if (!qbits && !apply) {  // binary32 sums, one message or several
        if (L.ntiles > 0) {
            ok(launch_dependent(k_dec_sum, sum_grid, kSumThreads, s, a));
            ++launches;
        }
    } else if (W == 1 && !apply) {
        // one message of integers: its positions are distinct, so the sum kernel's single-token
        // path (one dequantization per value, +0 elsewhere) is the whole decode
        if (L.ntiles > 0) {
            ok(launch_dependent(k_dec_sum, sum_grid, kSumThreads, s, a));
            ++launches;
        }
    } else if (W == 1) {  // the step from one message: one scattered update per value
        if (L.sum_T > 0) {
            ok(launch_dependent(k_dec_scatter1, (L.sum_T + kThreads - 1) / kThreads, kThreads, s,
                                a));
            ++launches;
        }
    } else if (L.ntiles > 0) {
        if (qbits)
            ok(launch_dependent(k_dec_tiles<true>, L.ntiles, kThreads, s, a));
        else
            ok(launch_dependent(k_dec_tiles<false>, L.ntiles, kThreads, s, a));
        ++launches;
    }
    if (e != cudaSuccess) return DGC_ECUDA;
    dgc_internal_count_launches(launches);
    if (cudaPeekAtLastError() != cudaSuccess) {
        cudaGetLastError();
        return DGC_ECUDA;
    }
    return DGC_OK;
}
}  // namespace

extern "C" int dgc_decode_accumulate_dev(const uint8_t* const* streams,
                                         const uint64_t* stream_bytes, const uint64_t* max_bytes,
                                         int32_t W, float* dense, int64_t n, int32_t accumulate,
                                         int32_t* status, void* ws, size_t ws_bytes,
                                         dgc_stream_t stream) {
    if (W > 0 && !stream_bytes) return DGC_EINVAL;
    return decode_impl(streams, max_bytes, W, dense, n, accumulate, 0, 0.0f, 0, 0.0f, status, ws,
                       ws_bytes, stream, stream_bytes);
}

extern "C" int dgc_decode_apply_dev(const uint8_t* const* streams, const uint64_t* stream_bytes,
                                    const uint64_t* max_bytes, int32_t W, float* w, int64_t n,
                                    float lr, int32_t* status, void* ws, size_t ws_bytes,
                                    dgc_stream_t stream) {
    if (W > 0 && !stream_bytes) return DGC_EINVAL;
    if (!std::isfinite(lr) || std::signbit(lr)) return DGC_EINVAL;
    return decode_impl(streams, max_bytes, W, w, n, 0, 1, lr, 0, 0.0f, status, ws, ws_bytes,
                       stream, stream_bytes);
}

extern "C" int dgc_decode_accumulate(const uint8_t* const* streams, const uint64_t* stream_bytes,
                                     int32_t W, float* dense, int64_t n, int32_t accumulate,
                                     int32_t* status, void* ws, size_t ws_bytes,
                                     dgc_stream_t stream) {
    return decode_impl(streams, stream_bytes, W, dense, n, accumulate, 0, 0.0f, 0, 0.0f, status,
                       ws, ws_bytes, stream);
}

extern "C" int dgc_decode_apply(const uint8_t* const* streams, const uint64_t* stream_bytes,
                                int32_t W, float* w, int64_t n, float lr, int32_t* status,
                                void* ws, size_t ws_bytes, dgc_stream_t stream) {
    if (!std::isfinite(lr) || std::signbit(lr)) return DGC_EINVAL;
    return decode_impl(streams, stream_bytes, W, w, n, 0, 1, lr, 0, 0.0f, status, ws, ws_bytes,
                       stream);
}

namespace {
int check_quant(int32_t W, int32_t bits, float alpha) {
    if ((bits != 8 && bits != 16) || !std::isfinite(alpha) || !(alpha > 0.0f)) return DGC_EINVAL;
    if (W > 65536) return DGC_EUNSUPPORTED;  // keeps every integer sum below 2^31
    return DGC_OK;
}
}  // namespace

extern "C" int dgc_decode_accumulate_quant(const uint8_t* const* streams,
                                           const uint64_t* stream_bytes, int32_t W, int32_t bits,
                                           float alpha, float* dense, int64_t n,
                                           int32_t accumulate, int32_t* status, void* ws,
                                           size_t ws_bytes, dgc_stream_t stream) {
    if (W < 0) return DGC_EINVAL;
    const int rc = check_quant(W, bits, alpha);
    if (rc) return rc;
    return decode_impl(streams, stream_bytes, W, dense, n, accumulate, 0, 0.0f, bits, alpha,
                       status, ws, ws_bytes, stream);
}

extern "C" int dgc_decode_apply_quant(const uint8_t* const* streams, const uint64_t* stream_bytes,
                                      int32_t W, int32_t bits, float alpha, float* w, int64_t n,
                                      float lr, int32_t* status, void* ws, size_t ws_bytes,
                                      dgc_stream_t stream) {
    if (W < 0 || !std::isfinite(lr) || std::signbit(lr)) return DGC_EINVAL;
    const int rc = check_quant(W, bits, alpha);
    if (rc) return rc;
    return decode_impl(streams, stream_bytes, W, w, n, 0, 1, lr, bits, alpha, status, ws,
                       ws_bytes, stream);
}

extern "C" int dgc_sum_shared_workspace(int32_t W, size_t* bytes) {
    if (!bytes || W < 0) return DGC_EINVAL;
    *bytes = align256(sizeof(float*) * (size_t)(W > 0 ? W : 1));
    return DGC_OK;
}

extern "C" int dgc_sum_shared(const float* const* vals, int32_t W, const int64_t* count,
                              int64_t max_count, float* out, int32_t* status, void* ws,
                              size_t ws_bytes, dgc_stream_t stream) {
    if (W < 0 || max_count < 0 || !count || !status || !ws) return DGC_EINVAL;
    if (max_count > 0 && !out) return DGC_EINVAL;
    if (W > 0 && !vals) return DGC_EINVAL;
    for (int w = 0; w < W; ++w)
        if (!vals[w] || ((uintptr_t)vals[w] & 3u) != 0) return DGC_EINVAL;
    if (((uintptr_t)ws & 255u) != 0) return DGC_EINVAL;
    size_t need;
    dgc_sum_shared_workspace(W, &need);
    if (ws_bytes < need) return DGC_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the pointer table goes to the device with the call (a pageable copy: staged before this
    // function returns, so the host array may go away)
    if (W > 0 && cudaMemcpyAsync(ws, vals, sizeof(float*) * (size_t)W, cudaMemcpyHostToDevice,
                                 s) != cudaSuccess)
        return DGC_ECUDA;
    const int sms = dgc_internal_sm_count();
    if (sms <= 0) return DGC_ECUDA;
    const unsigned grid = (unsigned)std::max<uint64_t>(
        1, std::min<uint64_t>((uint64_t)sms * 8, ((uint64_t)max_count + kThreads - 1) / kThreads));
    k_sum_shared<<<grid, kThreads, 0, s>>>(static_cast<const float* const*>(ws), W, count,
                                           (uint64_t)max_count, out, status);
    dgc_internal_count_launches(1);
    if (cudaPeekAtLastError() != cudaSuccess) {
        cudaGetLastError();
        return DGC_ECUDA;
    }
    return DGC_OK;
}
