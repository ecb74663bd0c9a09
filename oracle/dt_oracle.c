/*
 * dt_oracle.c -- CPU oracle for the same-device collective set.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; the two meet only through the seeded inputs that both read.
 *
 * Every function is the plain definition of one collective, written as a
 * slow single-threaded loop so that a reader can check it against the pages:
 *
 *   [DT]  "集合通信组件" (DTorch developer guide, collective communication
 *         component): §2.1 ThreadGroup interface, §2.3
 *         ThreadGroupSameDeviceBackend (the three-phase AllReduce: every rank
 *         publishes its tensor, rank 0 adds ranks 1..P-1 onto rank 0's tensor
 *         in ascending rank order, then hands the one result to every rank),
 *         §2.5 the placement-conversion matrix (P->R AllReduce, P->S
 *         ReduceScatter, S->R AllGather, S->S AllToAll).
 *   [PB]  "通信与互联（05）" (PyTorch communication stack: ProcessGroupNCCL and
 *         streams), §六.5: DDP flattens many gradients into 25 MB buckets.
 *   [BAR] "Barrier：仅信号（Signals Only）" (PyPTO): notify/wait barrier.
 *   [HP]  "异步融合 AllReduce 流水线优化" (MindSpore hyper-parallel issue
 *         #120), AllReduceParamGroup.wait_and_apply_grads: SUM all-reduce of
 *         the fused buffer, then divide each gradient view by the replicate
 *         world size when the op is AVG.
 *
 * Readings where the pages leave a step open (the library follows the same
 * readings, written independently):
 *   - Accumulation: fp32 for fp32 and bf16 inputs (bf16 widens exactly to
 *     fp32), wrapping 32-bit integer for int32; one rounding to bf16, round to
 *     nearest even, at the very end.  Ranks are combined in ascending order,
 *     rank 0 first, as the AllReduce of [DT] §2.3 does.
 *   - AVG: the fp32 sum divided by (float)P with one IEEE division [HP];
 *     AVG on int32 is unsupported.
 *   - MAX / MIN select one of the inputs: rank r's value replaces the running
 *     one when it is strictly greater (smaller) or is a NaN, so a NaN
 *     propagates and ties (including +0 / -0) keep the lower rank's value.
 *     The selected element's original bits are the result.
 *   - SUM_STEPWISE: the literal `result += DestGet(rank)` of [DT] §2.3, in
 *     which every add lands in the tensor's own dtype: ranks in ascending
 *     order, each fp32 add rounded back to bf16 before the next one.  For fp32
 *     and int32 it is SUM.
 *   - Bucket plan: greedy in the given order; a bucket is closed when adding
 *     the next tensor would take it past the cap; a tensor larger than the
 *     cap gets a bucket of its own.
 *
 * Compile with -O2 -std=c11 -ffp-contract=off: no fused multiply-add, no
 * extended precision (SSE2 on x86-64, plain fp on aarch64).
 */
#define _POSIX_C_SOURCE 200809L
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <sched.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_I32 = 2 };
enum { ORC_SUM = 0, ORC_AVG = 1, ORC_MAX = 2, ORC_MIN = 3, ORC_SUM_STEPWISE = 4 };
enum { ORC_OK = 0, ORC_INVALID = 1, ORC_UNSUPPORTED = 2 };

#define ORC_MAX_RANKS 64

/* ---------------------------------------------------------------- bf16 */

/* bf16 is the upper half of an IEEE binary32: widening appends 16 zero bits,
 * which is exact. */
float orc_bf16_to_f32(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* Narrow binary32 -> bf16 by IEEE round-to-nearest, ties to even, taken from
 * the definition: keep the upper 16 bits, look at the 16 discarded bits; more
 * than half an ulp rounds up, exactly half rounds to the even neighbour.  A
 * carry out of the mantissa bumps the exponent, which is also how a value
 * past the largest finite bf16 becomes infinity.  A NaN stays a NaN: its sign
 * and upper payload are kept and the quiet bit is set. */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    if ((bits & 0x7F800000u) == 0x7F800000u && (bits & 0x007FFFFFu) != 0)
        return (uint16_t)((bits >> 16) | 0x0040u);
    uint32_t upper = bits >> 16;
    uint32_t lower = bits & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;
    return (uint16_t)upper;
}

/* Array form of the narrowing above, for tests that sweep bit patterns. */
void orc_f32_to_bf16_array(const float *in, uint16_t *out, size_t n)
{
    for (size_t i = 0; i < n; i++)
        out[i] = orc_f32_to_bf16(in[i]);
}

/* --------------------------------------------------------- elementwise */

static size_t elem_size(int dtype)
{
    return dtype == ORC_BF16 ? 2 : 4;
}

static float load_f(int dtype, const void *base, size_t i)
{
    if (dtype == ORC_BF16) {
        uint16_t h;
        memcpy(&h, (const char *)base + 2 * i, 2);
        return orc_bf16_to_f32(h);
    }
    float f;
    memcpy(&f, (const char *)base + 4 * i, 4);
    return f;
}

static void store_f(int dtype, void *base, size_t i, float v)
{
    if (dtype == ORC_BF16) {
        uint16_t h = orc_f32_to_bf16(v);
        memcpy((char *)base + 2 * i, &h, 2);
    } else {
        memcpy((char *)base + 4 * i, &v, 4);
    }
}

static int32_t load_i(const void *base, size_t i)
{
    int32_t v;
    memcpy(&v, (const char *)base + 4 * i, 4);
    return v;
}

static int check_types(int dtype, int op)
{
    if (dtype != ORC_F32 && dtype != ORC_BF16 && dtype != ORC_I32)
        return ORC_INVALID;
    if (op < ORC_SUM || op > ORC_SUM_STEPWISE)
        return ORC_INVALID;
    if (dtype == ORC_I32 && op == ORC_AVG)
        return ORC_UNSUPPORTED;
    return ORC_OK;
}

/*
 * The one reduction every reducing collective is built from:
 *
 *   out[i] = narrow( scale( in_0[off+i] (+) in_1[off+i] (+) ... (+) in_{P-1}[off+i] ) )
 *
 * combined left to right in ascending rank order ([DT] §2.3: the result
 * starts as rank 0's tensor and ranks 1..P-1 are added onto it in turn).
 */
int orc_reduce(int dtype, int op, int P, const void *const *in, size_t in_offset,
               size_t n, void *out)
{
    int st = check_types(dtype, op);
    if (st != ORC_OK)
        return st;
    if (P < 1 || P > ORC_MAX_RANKS || (n > 0 && (!in || !out)))
        return ORC_INVALID;

    for (size_t i = 0; i < n; i++) {
        size_t k = in_offset + i;
        if (dtype == ORC_I32) {
            int32_t acc = load_i(in[0], k);
            for (int r = 1; r < P; r++) {
                int32_t x = load_i(in[r], k);
                if (op == ORC_SUM || op == ORC_SUM_STEPWISE)
                    acc = (int32_t)((uint32_t)acc + (uint32_t)x);   /* wraps mod 2^32 */
                else if (op == ORC_MAX)
                    acc = x > acc ? x : acc;
                else
                    acc = x < acc ? x : acc;
            }
            memcpy((char *)out + 4 * i, &acc, 4);
        } else if (op == ORC_MAX || op == ORC_MIN) {
            /* selection: remember which rank's element wins, copy its bits */
            int win = 0;
            float best = load_f(dtype, in[0], k);
            for (int r = 1; r < P; r++) {
                float x = load_f(dtype, in[r], k);
                int take = isnan(x) || (op == ORC_MAX ? x > best : x < best);
                if (take) {
                    best = x;
                    win = r;
                }
            }
            size_t es = elem_size(dtype);
            memcpy((char *)out + es * i, (const char *)in[win] + es * k, es);
        } else if (op == ORC_SUM_STEPWISE) {
            float acc = load_f(dtype, in[0], k);
            for (int r = 1; r < P; r++) {
                acc = acc + load_f(dtype, in[r], k);
                if (dtype == ORC_BF16)
                    acc = orc_bf16_to_f32(orc_f32_to_bf16(acc));   /* the += lands in bf16 */
            }
            store_f(dtype, out, i, acc);
        } else {
            float acc = load_f(dtype, in[0], k);
            for (int r = 1; r < P; r++)
                acc = acc + load_f(dtype, in[r], k);
            if (op == ORC_AVG)
                acc = acc / (float)P;
            store_f(dtype, out, i, acc);
        }
    }
    return ORC_OK;
}

/* P -> R ([DT] §2.1 AllReduce, §2.3): every rank receives the reduction of
 * all ranks' tensors.  out[q] may equal in[q] (in place): each element is
 * reduced into a temporary first. */
int orc_allreduce(int dtype, int op, int P, const void *const *in, void *const *out,
                  size_t n)
{
    int st = check_types(dtype, op);
    if (st != ORC_OK)
        return st;
    if (P < 1 || P > ORC_MAX_RANKS)
        return ORC_INVALID;
    size_t es = elem_size(dtype);
    unsigned char tmp[4];
    for (size_t i = 0; i < n; i++) {
        const void *col[ORC_MAX_RANKS];
        for (int r = 0; r < P; r++)
            col[r] = (const char *)in[r] + es * i;
        st = orc_reduce(dtype, op, P, col, 0, 1, tmp);
        if (st != ORC_OK)
            return st;
        for (int q = 0; q < P; q++)
            memcpy((char *)out[q] + es * i, tmp, es);
    }
    return ORC_OK;
}

/* P -> S(0) ([DT] §2.1 ReduceScatterTensor): every rank's input holds
 * P * recv_count elements; rank r receives the reduction, over all ranks, of
 * shard r = elements [r * recv_count, (r + 1) * recv_count). */
int orc_reduce_scatter(int dtype, int op, int P, const void *const *in,
                       void *const *out, size_t recv_count)
{
    int st = check_types(dtype, op);
    if (st != ORC_OK)
        return st;
    if (P < 1 || P > ORC_MAX_RANKS)
        return ORC_INVALID;
    for (int r = 0; r < P; r++) {
        st = orc_reduce(dtype, op, P, in, (size_t)r * recv_count, recv_count, out[r]);
        if (st != ORC_OK)
            return st;
    }
    return ORC_OK;
}

/* S(0) -> R ([DT] §2.1 AllGatherIntoTensor / AllGather with uneven shards):
 * every rank receives the concatenation along dim 0 of all ranks' shards in
 * ascending rank order; rank r holds rows[r] rows of row_bytes bytes and its
 * rows land at row offset rows[0] + ... + rows[r-1]. */
int orc_all_gather(int P, const void *const *in, void *const *out, const size_t *rows,
                   size_t row_bytes)
{
    if (P < 1 || P > ORC_MAX_RANKS || !rows)
        return ORC_INVALID;
    for (int q = 0; q < P; q++) {
        size_t offset_rows = 0;
        for (int r = 0; r < P; r++) {
            const unsigned char *src = in[r];
            unsigned char *dst = (unsigned char *)out[q] + offset_rows * row_bytes;
            for (size_t b = 0; b < rows[r] * row_bytes; b++)
                dst[b] = src[b];
            offset_rows += rows[r];
        }
    }
    return ORC_OK;
}

/* The one concatenation of the AllGather above, written to a single buffer
 * (every rank's output holds exactly this). */
int orc_all_gather_one(int P, const void *const *in, void *out, const size_t *rows,
                       size_t row_bytes)
{
    if (P < 1 || P > ORC_MAX_RANKS || !rows)
        return ORC_INVALID;
    size_t offset_rows = 0;
    for (int r = 0; r < P; r++) {
        const unsigned char *src = in[r];
        unsigned char *dst = (unsigned char *)out + offset_rows * row_bytes;
        for (size_t b = 0; b < rows[r] * row_bytes; b++)
            dst[b] = src[b];
        offset_rows += rows[r];
    }
    return ORC_OK;
}

/* S -> S ([DT] §2.1 AllToAll, split and concatenated along dim 0): rank i's
 * input is P chunks of chunk_bytes; chunk j goes to rank j, which stacks the
 * chunks it receives in ascending source rank:
 *   out_j[i * c + k] = in_i[j * c + k]. */
int orc_all_to_all(int P, const void *const *in, void *const *out, size_t chunk_bytes)
{
    if (P < 1 || P > ORC_MAX_RANKS)
        return ORC_INVALID;
    for (int j = 0; j < P; j++)
        for (int i = 0; i < P; i++) {
            const unsigned char *src = (const unsigned char *)in[i] + (size_t)j * chunk_bytes;
            unsigned char *dst = (unsigned char *)out[j] + (size_t)i * chunk_bytes;
            for (size_t k = 0; k < chunk_bytes; k++)
                dst[k] = src[k];
        }
    return ORC_OK;
}

/* R -> S ([DT] §2.1 ReplicateToShard, §2.5 placement matrix R -> S): every
 * rank holds the whole tensor (rows x row_bytes); the rows split evenly into P
 * blocks and rank r keeps block shard_idx[r] (its own rank when shard_idx is
 * NULL). */
int orc_replicate_to_shard(int P, const void *const *in, void *const *out, const int *shard_idx,
                           size_t rows, size_t row_bytes)
{
    if (P < 1 || P > ORC_MAX_RANKS || rows % (size_t)P)
        return ORC_INVALID;
    size_t block = rows / (size_t)P * row_bytes;
    for (int r = 0; r < P; r++) {
        int sidx = shard_idx ? shard_idx[r] : r;
        if (sidx < 0 || sidx >= P)
            return ORC_INVALID;
        const unsigned char *src = (const unsigned char *)in[r] + (size_t)sidx * block;
        unsigned char *dst = out[r];
        for (size_t b = 0; b < block; b++)
            dst[b] = src[b];
    }
    return ORC_OK;
}

/* S -> R as a vector ([DT] §2.1 AllGatherIntoVec): every rank keeps every
 * rank's shard as a tensor of its own: out[q * P + r] is rank r's shard as
 * received by rank q (rows[r] rows of row_bytes). */
int orc_all_gather_into_vec(int P, const void *const *in, void *const *out, const size_t *rows,
                            size_t row_bytes)
{
    if (P < 1 || P > ORC_MAX_RANKS || !rows)
        return ORC_INVALID;
    for (int q = 0; q < P; q++)
        for (int r = 0; r < P; r++) {
            const unsigned char *src = in[r];
            unsigned char *dst = out[q * P + r];
            for (size_t b = 0; b < rows[r] * row_bytes; b++)
                dst[b] = src[b];
        }
    return ORC_OK;
}

/* S(src_dim) -> S(dest_dim) ([DT] §2.1 AllToAll(input, srcDim, destDim),
 * §2.5 S -> S) for 2-D tensors of R x C elements of es bytes, row-major.
 * Rank i splits its tensor X_i along dest_dim into P equal parts; part j goes
 * to rank j, which concatenates the parts it receives along src_dim in
 * ascending source rank.  A part is h x w (h = R/P or R, w = C or C/P); rank
 * j's output is (P h) x w when src_dim is 0, h x (P w) when it is 1. */
int orc_all_to_all_2d(int P, const void *const *in, void *const *out, size_t R, size_t C,
                      size_t es, int src_dim, int dest_dim)
{
    if (P < 1 || P > ORC_MAX_RANKS || (src_dim != 0 && src_dim != 1) ||
        (dest_dim != 0 && dest_dim != 1))
        return ORC_INVALID;
    if ((dest_dim == 0 && R % (size_t)P) || (dest_dim == 1 && C % (size_t)P))
        return ORC_INVALID;
    size_t h = dest_dim == 0 ? R / P : R;
    size_t w = dest_dim == 1 ? C / P : C;
    size_t out_rows = src_dim == 0 ? (size_t)P * h : h;
    size_t out_cols = src_dim == 1 ? (size_t)P * w : w;
    for (int j = 0; j < P; j++)
        for (size_t a = 0; a < out_rows; a++)
            for (size_t b = 0; b < out_cols; b++) {
                /* which source rank, and where inside its part */
                size_t i = src_dim == 0 ? a / h : b / w;
                size_t pa = src_dim == 0 ? a % h : a;
                size_t pb = src_dim == 1 ? b % w : b;
                /* the part is block j of X_i along dest_dim */
                size_t xa = pa + (dest_dim == 0 ? (size_t)j * h : 0);
                size_t xb = pb + (dest_dim == 1 ? (size_t)j * w : 0);
                const unsigned char *src = (const unsigned char *)in[i] + (xa * C + xb) * es;
                unsigned char *dst = (unsigned char *)out[j] + (a * out_cols + b) * es;
                for (size_t k = 0; k < es; k++)
                    dst[k] = src[k];
            }
    return ORC_OK;
}

/* Bucket plan ([PB] §六.5: gradients are gathered into buckets of at most
 * bucket_cap bytes before one all-reduce per bucket).  Greedy in the given
 * order; writes bucket_of[t] and returns the number of buckets in *n_buckets. */
int orc_bucket_plan(const size_t *counts, size_t T, size_t elem_bytes, size_t cap_bytes,
                    size_t *bucket_of, size_t *n_buckets)
{
    if (!n_buckets || (T > 0 && (!counts || !bucket_of)) || elem_bytes == 0 || cap_bytes == 0)
        return ORC_INVALID;
    size_t b = 0, filled = 0;
    for (size_t t = 0; t < T; t++) {
        size_t bytes = counts[t] * elem_bytes;
        if (filled > 0 && filled + bytes > cap_bytes) {
            b++;
            filled = 0;
        }
        bucket_of[t] = b;
        filled += bytes;
    }
    *n_buckets = T > 0 ? b + 1 : 0;
    return ORC_OK;
}

/* Fused gradient-bucket all-reduce ([HP] wait_and_apply_grads): for every
 * tensor t and rank p, grads[t * P + p] is rank p's gradient t; each one is
 * replaced in place by the all-reduce (SUM, or SUM then divide by P for AVG)
 * of gradient t over the ranks.  Bucketing only groups the work, so the
 * result does not depend on the plan. */
int orc_bucket_allreduce(int dtype, int op, int P, void *const *grads, const size_t *counts,
                         size_t T)
{
    if (dtype != ORC_F32 && dtype != ORC_BF16)
        return ORC_UNSUPPORTED;
    if (op != ORC_SUM && op != ORC_AVG)
        return ORC_UNSUPPORTED;
    if (P < 1 || P > ORC_MAX_RANKS)
        return ORC_INVALID;
    for (size_t t = 0; t < T; t++) {
        const void *in[ORC_MAX_RANKS];
        for (int p = 0; p < P; p++)
            in[p] = grads[t * (size_t)P + p];
        int st = orc_allreduce(dtype, op, P, in, grads + t * (size_t)P, counts[t]);
        if (st != ORC_OK)
            return st;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------- barrier */

/*
 * Signal-window barrier of [BAR], run by P host threads on one window
 * win[P][P] (rank q's window is row block q; cell win[q*P + r] is "row r of
 * rank q's window").  Barrier number g (1-based) on rank r:
 *   notify: for every peer q != r, atomically add 1 to win[q][r]
 *           (row my_rank of the peer's window);
 *   wait:   for every src s != r, wait until win[r][s] >= g (the generation
 *           raises the threshold on every reuse of the window).
 * Each thread counts arrivals before it notifies and checks, once released,
 * that all P ranks had arrived at barrier g; *early_passes counts releases
 * that happened before that.  The window is left in win.
 */
typedef struct {
    int P, G, rank;
    _Atomic int32_t *win;
    _Atomic int32_t *arrived;   /* arrived[g-1]: ranks that reached barrier g */
    _Atomic int32_t *early;
} orc_bar_thread;

static void *orc_bar_run(void *arg)
{
    orc_bar_thread *t = arg;
    int P = t->P, r = t->rank;
    for (int g = 1; g <= t->G; g++) {
        atomic_fetch_add(&t->arrived[g - 1], 1);
        for (int q = 0; q < P; q++)
            if (q != r)
                atomic_fetch_add(&t->win[q * P + r], 1);
        for (int s = 0; s < P; s++) {
            if (s == r)
                continue;
            while (atomic_load(&t->win[r * P + s]) < g)
                sched_yield();
        }
        if (atomic_load(&t->arrived[g - 1]) != P)
            atomic_fetch_add(t->early, 1);
    }
    return NULL;
}

int orc_barrier_sim(int P, int G, int32_t *win_out, int32_t *early_passes)
{
    if (P < 1 || P > ORC_MAX_RANKS || G < 0 || G > 4096 || !win_out || !early_passes)
        return ORC_INVALID;
    static _Atomic int32_t win[ORC_MAX_RANKS * ORC_MAX_RANKS];
    static _Atomic int32_t arrived[4096];
    _Atomic int32_t early = 0;
    for (int i = 0; i < P * P; i++)
        atomic_store(&win[i], 0);
    for (int g = 0; g < G; g++)
        atomic_store(&arrived[g], 0);
    pthread_t th[ORC_MAX_RANKS];
    orc_bar_thread args[ORC_MAX_RANKS];
    for (int r = 0; r < P; r++) {
        args[r] = (orc_bar_thread){P, G, r, win, arrived, &early};
        if (pthread_create(&th[r], NULL, orc_bar_run, &args[r]) != 0) {
            for (int k = 0; k < r; k++)
                pthread_join(th[k], NULL);
            return ORC_INVALID;
        }
    }
    for (int r = 0; r < P; r++)
        pthread_join(th[r], NULL);
    for (int i = 0; i < P * P; i++)
        win_out[i] = atomic_load(&win[i]);
    *early_passes = atomic_load(&early);
    return ORC_OK;
}
