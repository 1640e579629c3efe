/*
 * dgc.h -- C ABI of libdgc: the per-worker gradient compressor of Deep Gradient Compression
 * (DGC) with AdaComp-style residual sparsification, its sparse message codec, and the
 * decode-and-sum aggregator, as CUDA kernels for NVIDIA GB300 (sm_103a).
 *
 * Sources, by page title and section:
 *   [DGC] "[Paper Review] Deep Gradient Compression: Reducing the Communication Bandwidth for
 *         Distributed Training": Abstract, Motivation & Objective, Proposed method (six
 *         bullets), Research questions (RQ4), Key findings.
 *   [ADA] "AdaComp : Adaptive Residual Gradient Compression for Data-Parallel Distributed
 *         Training": abstract and citation snippets.
 *   [SC]  the ScaleComp abstract (Scalable Sparsified Gradient Compression) on the first page
 *         of the sources, a taxoreview.com listing.
 *   [INT] "IntSGD: Adaptive Floatless Compression of Stochastic Gradients": abstract.
 *
 * Conventions for every call:
 *   - All array arguments are DEVICE pointers unless marked "host". The caller owns every
 *     buffer; the library allocates no device memory and frees none.
 *   - Work is enqueued on `stream` (a cudaStream_t; 0 is the legacy default stream). No call
 *     synchronizes with the device except dgc_read_status.
 *   - The return value reports errors that can be seen on the host before anything is
 *     enqueued (DGC_EINVAL, DGC_EUNSUPPORTED, DGC_ECORRUPT for malformed sizes); on such an
 *     error nothing is enqueued and no buffer is touched. DGC_ECUDA reports a launch the
 *     runtime refused; kernels of the call enqueued before it may have run, and the call's
 *     outputs are then invalid.
 *   - Errors that only the device can see are written to `*status` (an int32 in device
 *     memory): the first error wins and the library never clears it, so zero it before a
 *     sequence of calls and read it with dgc_read_status.
 *   - Scratch memory is the caller's `ws` buffer of at least the bytes the matching
 *     *_workspace query returns (256-byte aligned). A call may overwrite all of it; calls that
 *     share one workspace must be ordered (same stream, or synchronized). dgc_compress also
 *     keeps its sample positions there from one call to the next (they depend only on the seed
 *     and the segment layout); every call checks them against a tag and a checksum and
 *     rebuilds them when either differs, so using the workspace for anything else in between
 *     is safe and only costs that rebuild.
 *   - Indices are uint32: n must be below 2^32.
 *   - CUDA graphs: dgc_compress, dgc_compress_shared and dgc_encode enqueue kernels only
 *     (dgc_compress some of them as cooperative launches, dgc_encode its last two as
 *     programmatic dependent launches), so a stream capture of them replays as captured. Make one ordinary dgc_compress or dgc_compress_shared call on the
 *     device first (it sets the kernels' shared-memory attributes and reads the cooperative
 *     kernels' occupancy once per device). The decoders with host sizes read those sizes on
 *     the host at every call (and copy their table of messages from host memory when there are
 *     more than 96): capture the _dev decoders below instead. (This note does not cover
 *     dgc_compress_noalloc.)
 */
#ifndef DGC_H
#define DGC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dgc_stream_t; /* the same type as cudaStream_t */

enum {
    DGC_OK = 0,
    DGC_EINVAL = -1,       /* bad argument or segment table */
    DGC_ECAPACITY = -2,    /* an output buffer is too small */
    DGC_ECUDA = -3,        /* a CUDA call failed */
    DGC_ETIMEOUT = -4,     /* a bounded device-side wait gave up (results of the call invalid) */
    DGC_ECORRUPT = -5,     /* a message is malformed */
    DGC_EUNSUPPORTED = -6  /* a size the library does not handle (n >= 2^32) */
};

enum { DGC_SELECT_EXACT = 0, DGC_SELECT_SAMPLED = 1, DGC_SELECT_ADACOMP = 2 };
enum { DGC_FLAG_MASK_MOMENTUM = 1u };

/* Compressor settings. [DGC] Proposed method: momentum correction (momentum), local gradient
 * clipping (clip_norm), momentum factor masking (DGC_FLAG_MASK_MOMENTUM); [DGC] Abstract:
 * 99.9% sparsity; [DGC] RQ4: hierarchical thresholding (sample_ratio, reselect_factor);
 * [ADA] bin-local selection (bin_size); [SC] the low-pass filter in the local accumulation
 * (leak). */
typedef struct {
    uint32_t mode;          /* DGC_SELECT_EXACT, DGC_SELECT_SAMPLED or DGC_SELECT_ADACOMP */
    uint32_t flags;         /* DGC_FLAG_MASK_MOMENTUM: clear u where a value is sent */
    double sparsity;        /* fraction of each segment NOT sent, in [0, 1] */
    float momentum;         /* m in u <- m*u + g (finite) */
    float clip_norm;        /* per-segment L2 bound on g; <= 0 or +inf disables clipping */
    double sample_ratio;    /* sampled mode: fraction of each segment sampled, in (0, 1] */
    double reselect_factor; /* sampled mode: exact re-selection when |C| > factor*k, in [1,16] */
    uint64_t seed;          /* sampled mode: seed of the sample positions */
    uint32_t bin_size;      /* AdaComp mode: entries per bin, >= 1 (sparsity is not used) */
    float leak;             /* v <- fma(leak, v, u), in [0, 1]; 0 means 1: DGC's plain sum */
} dgc_params;

/* Per-segment statistics of one dgc_compress call. */
typedef struct {
    uint64_t k;          /* ceil(n_s * (1 - sparsity)); AdaComp: the number of bins */
    uint64_t candidates; /* sampled: |C| = #{i : |v_i| >= t}; exact and AdaComp: |S| */
    uint64_t sent;       /* |S| */
    uint32_t thresh_key; /* smallest |v| key (bits & 0x7FFFFFFF) among sent entries, or
                            0xFFFFFFFF when nothing was sent */
    uint32_t sample_key; /* sampled: the threshold key t; exact: 0 */
    uint32_t reselected; /* sampled: 1 if the exact re-selection ran */
    float clip_scale;    /* factor applied to g (1 when not clipped) */
    double clip_sumsq;   /* with clipping on: S, the squared L2 norm of the segment's g -- the
                            exact sum of the squares rounded once to binary64, ties to even
                            (NaN if an entry is NaN, else +inf if one is infinite); 0 with
                            clipping off */
} dgc_seg_stats;

/* ------------------------------------------------------------------------- compressor */

/* Bytes of workspace dgc_compress needs for n entries in nseg segments. */
int dgc_compress_workspace(int64_t n, int32_t nseg, const dgc_params* params, size_t* bytes);

/* Upper bound on the number of (index, value) pairs one dgc_compress call can emit; out_cap
 * must be at least this. Exact mode: sum of k; sampled mode: the re-selection rule bounds
 * |S| by reselect_factor * k per segment; AdaComp mode: n (ties can select a whole bin). */
int dgc_compress_max_out(int64_t n, int32_t nseg, const dgc_params* params, int64_t* max_out);

/* One compressor step over a flat buffer holding nseg segments (tensors), each compressed on
 * its own. [DGC] Proposed method, bullets 1 and 3-5; [DGC] RQ4; [ADA] abstract.
 *   1. k_s = ceil(n_s * (1 - sparsity)) per segment (integer arithmetic in parts per billion).
 *   2. If 0 < clip_norm < inf: scale_s = clip_norm / ||g_s|| when ||g_s|| > clip_norm (the
 *      squared norm S is the exact sum of the squares rounded once to binary64, ties to even:
 *      no order of summation shows; sqrt and the division correctly rounded in binary64, the
 *      quotient rounded once to binary32).
 *   3. u <- fma(m, u, g * scale); v <- v + u (binary32, round to nearest).
 *   4. S = the k_s largest |v| (ties to the lower index) in exact mode; in sampled mode
 *      t = the k_s'-th largest |v| among m_s = ceil(n_s * sample_ratio) positions drawn with
 *      SplitMix64 (seed), C = {|v| >= t}, and S = exact top-k_s of C when
 *      |C| > reselect_factor * k_s, else S = C. In AdaComp mode ([ADA] abstract and citation
 *      snippet) each segment is cut into bins of bin_size entries from its start (the last one
 *      shorter) and S = the entries whose |v| equals their bin's largest |v| (ties included;
 *      a bin whose largest |v| is 0 sends nothing).
 *   5. out_idx/out_val receive (i, v_i) for i in S in ascending i (segments in order), then
 *      v_i <- 0 and, with DGC_FLAG_MASK_MOMENTUM, u_i <- 0.
 * Arguments:
 *   g        device, n binary32, 16-byte aligned, read only (the fresh gradient)
 *   u, v     device, n binary32 each, 16-byte aligned, updated in place (momentum, residual)
 *   seg_off  device, nseg+1 int64: seg_off[0] = 0, seg_off[nseg] = n, non-decreasing (empty
 *            segments allowed). Checked on the device: a bad table sets *status = DGC_EINVAL
 *            and leaves every buffer but out_count and stats untouched.
 *   out_idx  device, out_cap uint32; out_val device, out_cap binary32; out_cap must be at
 *            least dgc_compress_max_out (else DGC_ECAPACITY is returned).
 *   out_count device, one int64: |S| summed over segments.
 *   stats    device, nseg dgc_seg_stats, or NULL.
 *   status   device, one int32 (see conventions).
 *   ws       device workspace, ws_bytes >= dgc_compress_workspace(...).
 * Every result is deterministic: the same inputs give the same bits on every run. */
int dgc_compress(const float* g, float* u, float* v, int64_t n, const int64_t* seg_off,
                 int32_t nseg, const dgc_params* params, uint32_t* out_idx, float* out_val,
                 int64_t out_cap, int64_t* out_count, dgc_seg_stats* stats, int32_t* status,
                 void* ws, size_t ws_bytes, dgc_stream_t stream);

/* dgc_compress for callers that cannot allocate device memory. The DGC and AdaComp pages have
 * no counterpart to this entry point: it exists for integration, not for the method.
 * Some callers cannot give the library a workspace at the point where they compress: their
 * framework's allocator owns all device memory and hands none out for a library's private use;
 * or they run while a CUDA graph is being captured, or in a loop where cudaMalloc (which may
 * synchronize the device) is not allowed; or they must not grow the process's device-memory
 * footprint once running. This variant takes dgc_compress's arguments without ws/ws_bytes and
 * works in a 16 MiB scratch array that the library holds on every GPU it is loaded on (created
 * when the library's device code loads on that GPU, kept until the process exits). It calls no
 * allocation routine.
 * Limit: the problem must fit the scratch, dgc_compress_workspace(n, nseg, params) <= 16 MiB --
 * about 2 million entries in one segment. A larger problem returns DGC_EUNSUPPORTED before
 * anything is enqueued; use dgc_compress with your own workspace instead.
 * The first call on each device looks the scratch address up with cudaGetSymbolAddress (which
 * may load the library's device code on that device); make that first call before any stream
 * capture. The address is kept with the identity of the CUDA context it was found in: after a
 * device reset (or a primary context released and created again) the next call finds a new
 * context and looks the address up again, so make that call outside stream capture too.
 * All later calls on the device reuse the same array; each call re-initialises every
 * part of it that it reads. Calls whose GPU work can overlap (streams without ordering between
 * them, several host threads) race on the shared array: the caller must serialize them. */
int dgc_compress_noalloc(const float* g, float* u, float* v, int64_t n, const int64_t* seg_off,
                         int32_t nseg, const dgc_params* params, uint32_t* out_idx,
                         float* out_val, int64_t out_cap, int64_t* out_count,
                         dgc_seg_stats* stats, int32_t* status, dgc_stream_t stream);

/* One index set for all learners. [SC] (the ScaleComp abstract, first page): a commutative
 * compressor keeps each learner's traffic independent of the number of learners and works with
 * all-reduce. This library's reading: every learner sends its accumulator at the same index set
 * S, so the learners' value vectors add up position by position. Which learner chooses S is the
 * caller's choice (for instance one learner in turn, with dgc_compress); the others then call
 * dgc_compress_shared with that S, and dgc_sum_shared adds the value vectors.
 *
 * One step at the given S: clipping and accumulation exactly as dgc_compress (same params; mode,
 * sparsity and the sample settings are not used), then out_val[j] = v[idx[j]] for j < *count,
 * and each sent entry leaves the accumulator (v <- 0, u <- 0 with masking).
 *   idx, count  device; idx strictly ascending and below n, 0 <= *count <= max_count, else
 *               *status = DGC_EINVAL and u, v and out_val are left as they were
 *   out_val     device, max_count binary32
 *   ws          dgc_compress_workspace(n, nseg, params) bytes suffice
 * Other arguments and errors as dgc_compress. */
int dgc_compress_shared(const float* g, float* u, float* v, int64_t n, const int64_t* seg_off,
                        int32_t nseg, const dgc_params* params, const uint32_t* idx,
                        const int64_t* count, int64_t max_count, float* out_val, int32_t* status,
                        void* ws, size_t ws_bytes, dgc_stream_t stream);

/* ------------------------------------------------------------------------------ codec */

/* Message format, [DGC] Proposed method, bullet 2 (each sent value a 32-bit word, each run of
 * zeros before it a 16-bit length); the byte layout is this library's reading:
 *   bytes 0..31: "DGC1", u16 version = 1, u16 flags = 0, u64 n, u64 T, u64 nnz (little-endian)
 *   then T binary32 values, then T u16 runs, then zero bytes up to a multiple of 4.
 * Entry j skips r = idx_j - idx_{j-1} - 1 zeros (idx_{-1} = -1); a skip of 65535 or more is
 * written as escape tokens (run 0xFFFF, value bits 0; each skips 65535 zeros and places no
 * value) followed by the entry's token with the remainder. Size = 32 + 6T (+2 when T is odd). */

/* Largest message dgc_encode can produce for at most max_count entries of an n-vector. */
int dgc_encode_max_bytes(int64_t max_count, int64_t n, uint64_t* bytes);

/* Bytes of workspace dgc_encode needs. */
int dgc_encode_workspace(int64_t max_count, size_t* bytes);

/* Encode count (device int64, at most max_count) ascending indices idx (device uint32) with
 * values val (device binary32) of an n-vector into out (device, out_cap bytes, 16-byte
 * aligned). *out_bytes (device u64) receives the message size. Indices that are not strictly
 * ascending or not below n set *status = DGC_EINVAL; a message larger than out_cap sets
 * DGC_ECAPACITY (*out_bytes still receives the size; out is not written). */
int dgc_encode(const uint32_t* idx, const float* val, const int64_t* count, int64_t max_count,
               int64_t n, uint8_t* out, uint64_t out_cap, uint64_t* out_bytes, int32_t* status,
               void* ws, size_t ws_bytes, dgc_stream_t stream);

/* Integer-valued messages (version 2). [ADA] abstract: AdaComp sends the selected residues
 * sparse and quantized; the IntSGD page, abstract: each learner scales its vector by a number
 * every learner knows and rounds to integers, so no float crosses the wire. The pages give no
 * bit format ([INT] is the IntSGD abstract); this library's reading:
 *   q_j = clamp(rint(alpha * val_j), -Q, Q), Q = 2^(bits-1) - 1, bits 8 or 16: one binary32
 *         multiply, rounding half to even, NaN to 0;
 *   the residual takes back what q_j does not carry: v[idx_j] = val_j - (float)q_j / alpha
 *         (one binary32 divide, one subtract);
 *   layout: "DGC1", u16 version 2, u16 bits, u64 n, u64 T, binary32 alpha, u32 nnz; T integers
 *         of `bits` bits (escape tokens carry 0); one zero byte when that ends on an odd offset;
 *         T u16 runs as in version 1; nothing after them, so a message's size fixes its T.
 * Receivers add the integers exactly (the order cannot change the sum) and divide once:
 * value_i = (float)S_i / alpha. alpha and bits are settings every learner and receiver share. */

/* Encode count (device int64, at most max_count) ascending indices idx with values val as a
 * version-2 message, as dgc_encode does for version 1 (same workspace, same errors; the message
 * is never larger than dgc_encode_max_bytes). v (device, n binary32, or NULL) is the residual:
 * v[idx_j] is overwritten with val_j - (float)q_j / alpha, the compressor having left 0 there.
 * alpha must be finite and > 0, bits 8 or 16, else DGC_EINVAL. */
int dgc_encode_quant(const uint32_t* idx, const float* val, const int64_t* count,
                     int64_t max_count, int64_t n, float alpha, int32_t bits, float* v,
                     uint8_t* out, uint64_t out_cap, uint64_t* out_bytes, int32_t* status,
                     void* ws, size_t ws_bytes, dgc_stream_t stream);

/* ---------------------------------------------------------------------------- decoder */

/* Bytes of workspace dgc_decode_accumulate or dgc_decode_apply needs for W messages of the
 * given sizes (host). */
int dgc_decode_workspace(int32_t W, const uint64_t* stream_bytes, int64_t n, size_t* bytes);

/* Decode W messages and sum them into dense (device, n binary32): synchronous SGD adds up
 * every learner's update ([DGC] Abstract, Motivation). The sum runs in learner order 0..W-1,
 * one binary32 addition per received value, onto +0 (accumulate = 0) or onto dense's current
 * contents (accumulate = 1), so the result is bitwise deterministic.
 *   streams       host array of W device pointers (16-byte aligned)
 *   stream_bytes  host array of W sizes; a size that no message can have returns DGC_ECORRUPT
 * A message whose header (magic, version, n, T) or runs (a position at or past n) are wrong
 * sets *status = DGC_ECORRUPT and dense is left as it was; nothing is written outside
 * dense[0, n). */
int dgc_decode_accumulate(const uint8_t* const* streams, const uint64_t* stream_bytes,
                          int32_t W, float* dense, int64_t n, int32_t accumulate,
                          int32_t* status, void* ws, size_t ws_bytes, dgc_stream_t stream);

/* Decode W messages, sum them and take one plain SGD step on the weights w (device, n
 * binary32): s = the sum dgc_decode_accumulate would produce from +0 (learner order 0..W-1),
 * then w_i <- fma(-lr, s_i, w_i) with one rounding. [DGC] Abstract (distributed SGD) and
 * Proposed method (momentum correction keeps the velocity on each learner, so the messages
 * already carry the momentum-corrected update): the receiver's step is plain SGD. Fold any
 * 1/W average into lr.
 *   lr  finite, sign bit clear (+0 allowed); anything else returns DGC_EINVAL. Under that rule
 *       the update is the identity wherever no message lands, and those entries are not
 *       touched at all: no dense sum is written, w is read and written only at received
 *       positions.
 * Workspace: dgc_decode_workspace. Arguments and errors as for dgc_decode_accumulate; on
 * DGC_ECORRUPT w is left as it was. */
int dgc_decode_apply(const uint8_t* const* streams, const uint64_t* stream_bytes, int32_t W,
                     float* w, int64_t n, float lr, int32_t* status, void* ws, size_t ws_bytes,
                     dgc_stream_t stream);

/* The decoders with the message sizes in device memory. [DGC] Abstract (the learners' updates
 * are exchanged and summed): a message's size is known on the device once the message is there,
 * for instance after an all-gather of the sizes, or right after dgc_encode wrote it. These calls
 * take the sizes from there, so nothing waits for them on the host, and with at most 96 messages
 * the call enqueues only kernels (a memset as well when W = 0; its message table travels in
 * kernel parameters; every kernel after the first is a programmatic dependent launch, which may
 * start while the one ahead of it finishes), so it can be captured in a CUDA graph together with
 * dgc_compress and dgc_encode.
 *   stream_bytes  device, W uint64 sizes (8-byte aligned); dgc_encode's out_bytes fits.
 *   max_bytes     host, W upper bounds on those sizes (for instance dgc_encode_max_bytes of the
 *                 encoder's max_count); the workspace is laid out for them.
 * A size that no binary32 message can have, or that exceeds its bound, sets *status to
 * DGC_ECORRUPT and leaves dense (w) as it was, like any malformed message. Everything else --
 * arguments, order of the sum, results, errors -- as dgc_decode_accumulate / dgc_decode_apply.
 * Workspace: dgc_decode_workspace_bound(W, max_bytes, n). */
int dgc_decode_workspace_bound(int32_t W, const uint64_t* max_bytes, int64_t n, size_t* bytes);
int dgc_decode_accumulate_dev(const uint8_t* const* streams, const uint64_t* stream_bytes,
                              const uint64_t* max_bytes, int32_t W, float* dense, int64_t n,
                              int32_t accumulate, int32_t* status, void* ws, size_t ws_bytes,
                              dgc_stream_t stream);
int dgc_decode_apply_dev(const uint8_t* const* streams, const uint64_t* stream_bytes,
                         const uint64_t* max_bytes, int32_t W, float* w, int64_t n, float lr,
                         int32_t* status, void* ws, size_t ws_bytes, dgc_stream_t stream);

/* Workspace for the version-2 decoders: W messages of `bits`-bit values with the given sizes. */
int dgc_decode_workspace_quant(int32_t W, const uint64_t* stream_bytes, int64_t n, int32_t bits,
                               size_t* bytes);

/* Decode W version-2 messages whose values are `bits`-bit integers scaled by alpha. S_i = the
 * exact integer sum over the messages; dense_i = (float)S_i / alpha (accumulate = 0: every
 * entry, +0 where nothing landed), or dense_i + (float)S_i / alpha at the positions some message
 * reaches (accumulate = 1; one binary32 addition, other entries untouched). A message whose
 * version, width, alpha (bitwise), n or T differ from the call's sets *status = DGC_ECORRUPT and
 * leaves dense as it was. bits other than 8 or 16, or alpha not finite and > 0: DGC_EINVAL;
 * W > 65536: DGC_EUNSUPPORTED (so |S_i| < 2^31). Other arguments as dgc_decode_accumulate. */
int dgc_decode_accumulate_quant(const uint8_t* const* streams, const uint64_t* stream_bytes,
                                int32_t W, int32_t bits, float alpha, float* dense, int64_t n,
                                int32_t accumulate, int32_t* status, void* ws, size_t ws_bytes,
                                dgc_stream_t stream);

/* The SGD step of dgc_decode_apply with version-2 messages: w_i <- fma(-lr, (float)S_i / alpha,
 * w_i) where S_i != 0, w untouched elsewhere (where the step is the identity). Arguments and
 * errors as dgc_decode_apply and dgc_decode_accumulate_quant. */
int dgc_decode_apply_quant(const uint8_t* const* streams, const uint64_t* stream_bytes, int32_t W,
                           int32_t bits, float alpha, float* w, int64_t n, float lr,
                           int32_t* status, void* ws, size_t ws_bytes, dgc_stream_t stream);

/* Workspace for dgc_sum_shared: the table of W pointers. */
int dgc_sum_shared_workspace(int32_t W, size_t* bytes);

/* The sum of W learners' value vectors over one shared index set, the step an all-reduce would
 * take: out[j] = the learner-ordered sum from +0 of vals[w][j] (w = 0..W-1, one binary32 addition
 * each, the order the decoders use), for j < *count (device int64, 0 <= *count <= max_count,
 * else *status = DGC_EINVAL and out is not written).
 *   vals  host array of W device pointers (4-byte aligned), each to *count binary32
 *   out   device, max_count binary32; it may be one of vals only if that is vals[0] */
int dgc_sum_shared(const float* const* vals, int32_t W, const int64_t* count, int64_t max_count,
                   float* out, int32_t* status, void* ws, size_t ws_bytes, dgc_stream_t stream);

/* -------------------------------------------------------------------------- utilities */

/* Synchronize `stream`, then return the int32 at status_dev (or DGC_ECUDA). */
int dgc_read_status(const int32_t* status_dev, dgc_stream_t stream);

/* Static text for a status code. */
const char* dgc_status_string(int code);

/* Number of kernels this library has launched in this process (all calls, all threads). */
uint64_t dgc_launch_count(void);

/* Sets the current device's context limit cudaLimitMaxL2FetchGranularity (bytes, 0..128; a hint
 * to the L2 on how much to fetch from DRAM per miss). The sampled threshold gathers g, u and v
 * at scattered positions, one 4-byte word each; 64 (or 32) keeps each miss from pulling in a
 * whole 128-byte line and shortened a 1B-entry step by ~0.15 ms on GB300, with the streaming
 * kernels unchanged. The limit belongs to the calling process's context and applies to every
 * kernel it launches afterwards; the library never sets it on its own. Returns DGC_EINVAL for a
 * value out of range, DGC_ECUDA if the runtime refuses it. */
int dgc_set_l2_fetch_granularity(int32_t bytes);

/* Profiling hook for benchmarks: while begin and end are non-NULL, every dgc_compress and
 * dgc_compress_shared call records `begin` on its stream right before its streaming pass (the
 * kernel that touches all n entries) and `end` right after it. dgc_profile_stream_pass(NULL,
 * NULL) turns it off. The setting is process-wide and not synchronized between threads. */
typedef struct CUevent_st* dgc_event_t; /* the same type as cudaEvent_t */
void dgc_profile_stream_pass(dgc_event_t begin, dgc_event_t end);

/* Self-test of the bounded device-side wait used by every cross-block scan: launches one
 * block that waits on a flag nothing ever sets, with at most spin_limit polls, and must come
 * back with *status = DGC_ETIMEOUT. Returns the launch status. */
int dgc_selftest_wait_timeout(int32_t* status, uint32_t spin_limit, dgc_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DGC_H */
