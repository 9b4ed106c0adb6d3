// Host planner: lays out a tensor group into one flat buffer of m shard slices.
//
// "veScale-FSDP: Flexible and High-Performance FSDP at Scale", §5 Planning
// algorithm: minimise the per-shard size S over the tensor offsets l_t subject to
// unsharded blocks, contiguous tensor memory and balanced load, with the tensors
// in their default order (the order the pages adopt).  Written out:
//   (i)   l_t >= l_{t-1} + n_{t-1}            (order kept, padding between tensors)
//   (ii)  l_t and S are multiples of a        (alignment)
//   (iii) a boundary B_k with l_t < B_k < l_t + n_t has (B_k - l_t) % g_t == 0
//   (iv)  l_last + n_last <= B_m
// The pages' Algorithm 1 reasons per tensor over three cases: the tensor fits in
// one shard, it straddles neighbouring shards without containing a whole one,
// or it contains at least one whole shard.  This planner uses those cases in two
// places:
//   * to find, at a fixed S, the leftmost start of each tensor in O(1) per shard
//     visited (case 1: fits; case 2: the start must sit a multiple of g_t before
//     the next boundary; case 3: additionally S % g_t == 0 for even shards);
//   * to skip sizes S that case 3 rules out for every placement: a tensor with
//     n_t > 2S always contains two consecutive boundaries, so S % g_t == 0 is
//     necessary.  Skipping is exact: every skipped S is infeasible.
// Feasibility in S is not monotone (a larger S can move boundaries onto bad
// residues), so the sizes are scanned upward instead of bisected, and the result
// is the exact minimum over multiples of a.  At that S the greedy-leftmost
// offsets are returned; they are optimal at fixed S because an earlier end of
// tensor t can only widen the choices of tensor t+1.
#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <new>
#include <thread>

#include "dbuf_internal.h"

namespace {

using dbuf::Chunk;
using dbuf::QItem;
using dbuf::TensorDesc;

constexpr int64_t kMaxElems = int64_t(1) << 50;

int64_t gcd64(int64_t a, int64_t b) {
    while (b) {
        int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

struct Geometry {
    bool even;
    int m;
    int64_t U;
    const int64_t *c;  // prefix sums of the shares, c[0..m]

    int64_t B(int k) const { return even ? U * k : U * c[k]; }

    // Largest j in [0, m-1] with B(j) <= p (p < B(m)).
    int shard_of(int64_t p) const {
        if (even) {
            int64_t j = p / U;
            return j >= m ? m - 1 : int(j);
        }
        int lo = 0, hi = m;  // B(lo) <= p < B(hi)
        while (hi - lo > 1) {
            int mid = (lo + hi) >> 1;
            if (U * c[mid] <= p) lo = mid;
            else hi = mid;
        }
        return lo;
    }
};

struct TensorGeom {
    int64_t n;  // elements
    int64_t g;  // unit (clamped to n for indivisible tensors)
    int64_t L;  // lcm(a, g)
};

// Leftmost start >= p satisfying (ii)-(iii) for one tensor; a start with
// start + n > B(m) means the tensor no longer fits.
int64_t first_start(int64_t p, const TensorGeom &t, const Geometry &geo) {
    if (t.n == 0) return p;
    const int64_t Bm = geo.B(geo.m);
    for (;;) {
        if (p + t.n > Bm) return p;
        const int j = geo.shard_of(p);
        const int64_t end = geo.B(j + 1);
        if (p + t.n <= end) return p;          // case 1: inside shard j
        if (t.g >= t.n) { p = end; continue; } // one indivisible unit
        const int64_t q = end - ((end - p) / t.L) * t.L;
        if (q == end) { p = end; continue; }
        // case 2 holds at q; case 3 needs every later boundary on a unit edge.
        bool ok = true;
        if (geo.even) {
            if (q + t.n > end + geo.U && geo.U % t.g != 0) ok = false;
        } else {
            for (int k = j + 2; k < geo.m && geo.B(k) < q + t.n; ++k)
                if ((geo.B(k) - end) % t.g != 0) { ok = false; break; }
        }
        if (ok) return q;
        p = end;
    }
}

// Greedy-leftmost placement at unit size U; fills `off` and returns true when
// every tensor fits.  rem[t] = elements of tensors t.. (early exit).
bool place(const std::vector<TensorGeom> &ts, const std::vector<int64_t> &rem, int64_t a,
           const Geometry &geo, int64_t *off) {
    const int64_t Bm = geo.B(geo.m);
    int64_t pos = 0;
    const size_t n = ts.size();
    for (size_t t = 0; t < n; ++t) {
        const int64_t p = first_start(round_up(pos, a), ts[t], geo);
        if (p + rem[t] > Bm) return false;
        off[t] = p;
        pos = p + ts[t].n;
    }
    return true;
}

// Feasibility of unit size U, in O(crossed boundaries * log n) instead of O(n).
// Inside one shard no tensor meets a boundary, so the greedy offsets there are
// aligned prefix sums: a tensor starting at an aligned p is followed by one at
// p + roundup(n_t, a).  P[t] = sum of roundup(n_i, a) for i < t.  The first
// tensor that would run past the shard end is found by binary search
// (P[t] + n_t is non-decreasing in t) and placed by the three-case rule; the
// scan then continues after it.  Same verdict as place().
bool feasible(const std::vector<TensorGeom> &ts, const std::vector<int64_t> &P,
              const std::vector<int64_t> &rem, int64_t a, const Geometry &geo) {
    const int64_t Bm = geo.B(geo.m);
    const int n = int(ts.size());
    int t = 0;
    int64_t pos = 0;  // aligned start candidate of tensor t
    while (t < n) {
        if (pos + rem[t] > Bm) return false;
        if (rem[t] == 0) return true;  // only empty tensors left
        const int64_t end = geo.B(geo.shard_of(pos) + 1);
        // first t' >= t with pos + P[t'] - P[t] + n_t' > end
        int lo = t, hi = n;
        const int64_t base = pos - P[t];
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (base + P[mid] + ts[mid].n > end) hi = mid;
            else lo = mid + 1;
        }
        if (lo == n) return true;  // every remaining tensor fits in this shard
        const int64_t p0 = base + P[lo];
        const int64_t p = first_start(p0, ts[lo], geo);
        if (p + rem[lo] > Bm) return false;
        pos = round_up(p + ts[lo].n, a);
        t = lo + 1;
    }
    return true;
}

// Smallest S' >= S (multiple of a) with S' % g_t == 0 for every tensor that has
// n_t > 2 S' (even shards).  `thr` holds (floor((n_t-1)/2), g_t) sorted by
// threshold, descending: the constraint of t is active while S' <= threshold.
int64_t next_candidate(int64_t S, int64_t a, const std::vector<std::pair<int64_t, int64_t>> &thr) {
    S = round_up(S, a);
    for (;;) {
        int64_t L = a;
        int64_t lowest_active = -1;
        bool huge = false;
        for (const auto &tg : thr) {
            if (tg.first < S) break;
            lowest_active = tg.first;
            const int64_t g = tg.second;
            const int64_t d = gcd64(L, g);
            if (L / d > kMaxElems / g) { huge = true; break; }
            L = L / d * g;
        }
        if (lowest_active < 0) return S;
        if (!huge) {
            const int64_t S2 = round_up(S, L);
            if (S2 <= lowest_active) return S2;
        }
        S = round_up(lowest_active + 1, a);
    }
}

int validate(const dbuf_tensor_spec *specs, int32_t n, int32_t m, const int32_t *units,
             int64_t align) {
    if (n < 0 || m < 1 || align < 1 || align > (int64_t(1) << 30)) return DBUF_EINVAL;
    if (n > 0 && !specs) return DBUF_EINVAL;
    if (units)
        for (int k = 0; k < m; ++k)
            if (units[k] < 1 || units[k] > (1 << 20)) return DBUF_EINVAL;
    int64_t E = 0;
    for (int32_t t = 0; t < n; ++t) {
        const dbuf_tensor_spec &s = specs[t];
        if (s.rows < 0 || s.cols < 0 || s.gran_rows < 0 || s.reserved != 0) return DBUF_EINVAL;
        if (s.rows > kMaxElems || s.cols > kMaxElems) return DBUF_ERANGE;
        // block rows and block columns are indexed with 32-bit integers
        if (s.quant != DBUF_QUANT_NONE && (s.rows >= (int64_t(1) << 31) || s.cols >= (int64_t(1) << 31)))
            return DBUF_ERANGE;
        if (s.cols > 0 && s.rows > kMaxElems / s.cols) return DBUF_ERANGE;
        const int64_t numel = s.rows * s.cols;
        if (numel > kMaxElems - E) return DBUF_ERANGE;
        E += numel;
        if (s.quant < DBUF_QUANT_NONE || s.quant > DBUF_QUANT_INT8) return DBUF_EINVAL;
        if (s.quant != DBUF_QUANT_NONE) {
            if (s.qblock_rows < 0 || s.qblock_cols < 0) return DBUF_EINVAL;
            const int64_t qr = s.qblock_rows > 0 ? s.qblock_rows : std::max<int64_t>(s.rows, 1);
            const bool cuttable = s.gran_rows > 0 && s.gran_rows < s.rows;
            if (cuttable && s.gran_rows % qr != 0) return DBUF_EINVAL;
            // elements of one block are counted with 32-bit integers
            const int64_t qc = s.qblock_cols > 0 ? s.qblock_cols : std::max<int64_t>(s.cols, 1);
            if (std::min(qr, std::max<int64_t>(s.rows, 1)) * std::min(qc, std::max<int64_t>(s.cols, 1)) >=
                (int64_t(1) << 31))
                return DBUF_ERANGE;
        }
    }
    return DBUF_OK;
}

void build_tables(dbuf_plan_t *p) {
    const int32_t n = p->n;
    p->tdesc.assign(n, TensorDesc{});
    p->scale_offsets.assign(n, 0);
    p->chunks.clear();
    p->row_items.clear();
    p->tile_items.clear();
    p->pipe_items.clear();
    p->pipe_tensors.clear();
    p->pipe_item_start.assign(1, 0);
    p->opt_items.clear();
    p->opt_plain.clear();
    p->p8_items.clear();
    p->p8_tensors.clear();
    p->p8_item_start.assign(1, 0);
    p->big_items.clear();
    p->big_tensors.clear();
    p->big_item_start.assign(1, 0);
    std::vector<dbuf::OptItem> p8_opt;  // register-kernel items of p8 tensors (the fallback)
    p->state_offsets.assign(n, -1);
    int64_t s_off = 0, st_off = 0;
    for (int32_t t = 0; t < n; ++t) {
        const dbuf_tensor_spec &s = p->specs[t];
        TensorDesc &d = p->tdesc[t];
        d.buf_off = p->offsets[t];
        d.src_off = p->src_offsets.empty() ? 0 : p->src_offsets[t];
        d.rows = s.rows;
        d.cols = s.cols;
        d.numel = s.rows * s.cols;
        d.quant = s.quant;
        d.qrows = int32_t(std::max<int64_t>(1, s.qblock_rows > 0 ? s.qblock_rows : s.rows));
        d.qcols = int32_t(std::max<int64_t>(1, s.qblock_cols > 0 ? s.qblock_cols : s.cols));
        d.nbc = s.cols > 0 ? int32_t((s.cols + d.qcols - 1) / d.qcols) : 0;
        d.scale_off = s_off;
        p->scale_offsets[t] = s_off;
        d.chunk_begin = int32_t(p->chunks.size());
        for (int64_t o = 0; o < d.numel; o += dbuf::kChunkElems)
            p->chunks.push_back(Chunk{o, t, int32_t(std::min(dbuf::kChunkElems, d.numel - o))});
        d.chunk_end = int32_t(p->chunks.size());
        d.state_off = -1;
        if (s.quant == DBUF_QUANT_NONE) {
            // compact fp32 moments of the 8-bit optimizer, 16-byte aligned starts
            d.state_off = st_off;
            p->state_offsets[t] = st_off;
            st_off += (d.numel + 3) / 4 * 4;
            for (int32_t c = d.chunk_begin; c < d.chunk_end; ++c) p->opt_plain.push_back(c);
        }
        if (s.quant != DBUF_QUANT_NONE && d.numel > 0) {
            const int64_t nbr = (s.rows + d.qrows - 1) / d.qrows;
            const int64_t nb = nbr * d.nbc;
            {
                // 8-bit optimizer items: the fewest threads per block that keep the
                // block in registers (units of 4 elements when rows and block
                // widths allow vector access), 256 threads and a recompute pass for
                // larger blocks; about kOptItemElems elements per item.
                const int64_t be = int64_t(d.qrows) * d.qcols;
                const bool vec = d.qcols % 4 == 0 && s.cols % 4 == 0 && d.buf_off % 4 == 0;
                const int64_t units = vec ? be / 4 : be;
                int lanes = 4;
                while (lanes < 256 && units > int64_t(lanes) * dbuf::kOptUnitsPerLane) lanes *= 2;
                const int64_t groups = 256 / lanes;
                int64_t per = std::max<int64_t>(1, dbuf::kOptItemElems / std::max<int64_t>(1, be));
                per = std::max<int64_t>(groups, (per + groups - 1) / groups * groups);
                per = std::min<int64_t>(per, 16384);
                // The pipelined kernel takes power-of-two blocks of at most one stage
                // (and at least one unit of every compute thread of a block group)
                // whose rows are 16-byte aligned in every buffer (fp32 and codes).
                auto pow2 = [](int64_t x) { return x > 0 && (x & (x - 1)) == 0; };
                const bool p8 = pow2(d.qrows) && pow2(d.qcols) && d.qcols >= 16 && d.qcols <= 256 &&
                                be <= dbuf::kP8StageElems && be >= 4 * dbuf::kP8UnitsPerThread &&
                                s.cols % 16 == 0 &&
                                d.buf_off % 16 == 0 && s.rows < (int64_t(1) << 31) &&
                                s.cols < (int64_t(1) << 31);
                // Blocks of kBigBlockElems (two stages) take the big-block kernel under
                // the same alignment rules, with box dimensions of at most 256.
                const bool big = pow2(d.qrows) && pow2(d.qcols) && be == dbuf::kBigBlockElems &&
                                 d.qcols >= 64 && d.qcols <= 256 && d.qrows <= 256 &&
                                 s.cols % 16 == 0 && d.buf_off % 16 == 0 &&
                                 s.rows < (int64_t(1) << 31) && s.cols < (int64_t(1) << 31);
                std::vector<dbuf::OptItem> &dst = (p8 || big) ? p8_opt : p->opt_items;
                for (int64_t b = 0; b < nb; b += per)
                    dst.push_back(dbuf::OptItem{t, int32_t(b / d.nbc), int32_t(b % d.nbc),
                                                int16_t(std::min(per, nb - b)), int16_t(lanes)});
                if (p8) {
                    // the slot within its launch of at most kP8MaxTensors tensors
                    const int32_t slot = int32_t(p->p8_tensors.size() % dbuf::kP8MaxTensors);
                    p->p8_tensors.push_back(t);
                    const int64_t nblk = dbuf::kP8StageElems / be;
                    const int64_t K = std::min<int64_t>(256 / d.qcols, nblk);
                    const int64_t Rb = nblk / K;
                    for (int64_t bi = 0; bi < nbr; bi += Rb)
                        for (int64_t bj = 0; bj < d.nbc; bj += K)
                            p->p8_items.push_back(
                                dbuf::P8Item{slot, t, int32_t(bi), int32_t(bj)});
                    p->p8_item_start.push_back(p->p8_items.size());
                }
                if (big) {
                    const int32_t slot = int32_t(p->big_tensors.size() % dbuf::kP8MaxTensors);
                    p->big_tensors.push_back(t);
                    for (int64_t bi = 0; bi < nbr; ++bi)
                        for (int64_t bj = 0; bj < d.nbc; ++bj)
                            p->big_items.push_back(
                                dbuf::P8Item{slot, t, int32_t(bi), int32_t(bj)});
                    p->big_item_start.push_back(p->big_items.size());
                }
            }
            if (d.qrows == 1) {
                for (int64_t b = 0; b < nb; b += dbuf::kRowItemBlocks)
                    p->row_items.push_back(dbuf::RowItem{
                        t, int32_t(b / d.nbc), int32_t(b % d.nbc),
                        int32_t(std::min<int64_t>(dbuf::kRowItemBlocks, nb - b))});
            } else {
                // Tiles a 2-D tensor map can fetch (rows and tile widths multiples of
                // 16 bytes at a 16-byte-aligned tensor offset) go to the pipelined
                // kernel, which takes kPipeMaxTensors tensors per launch (an item
                // carries its tensor's slot within the launch); the rest to the
                // register-tile kernel.
                const bool pipe = d.qrows <= dbuf::kPipeMaxRows && d.qcols <= dbuf::kPipeMaxCols &&
                                  d.qcols % 4 == 0 && s.cols % 4 == 0 && d.buf_off % 4 == 0 &&
                                  s.rows < (int64_t(1) << 31) && s.cols < (int64_t(1) << 31);
                const int32_t slot =
                    pipe ? int32_t(p->pipe_tensors.size() % dbuf::kPipeMaxTensors) : -1;
                if (pipe) p->pipe_tensors.push_back(t);
                for (int64_t b = 0; b < nb; ++b) {
                    if (pipe)
                        p->pipe_items.push_back(
                            dbuf::TileItem{t, int32_t(b / d.nbc), int32_t(b % d.nbc), slot});
                    else
                        p->tile_items.push_back(QItem{b, t, 1});
                }
                if (pipe) p->pipe_item_start.push_back(p->pipe_items.size());
            }
            s_off += nb;
        }
    }
    p->n_scales = s_off;
    p->n_state = st_off;
    p->n_opt_rest = p->opt_items.size();
    p->opt_items.insert(p->opt_items.end(), p8_opt.begin(), p8_opt.end());

    // gather / scatter pieces: each tensor's chunks cut again at shard bounds
    p->pieces.clear();
    int32_t k = 0;
    for (int32_t t = 0; t < n; ++t) {
        const int64_t l = p->offsets[t], numel = p->tdesc[t].numel;
        int64_t i = 0;
        while (i < numel) {
            const int64_t pos = l + i;
            while (k + 1 < p->m && p->bounds[k + 1] <= pos) ++k;
            int64_t end = std::min(numel, (i / dbuf::kChunkElems + 1) * dbuf::kChunkElems);
            end = std::min(end, p->bounds[k + 1] - l);
            p->pieces.push_back(dbuf::Piece{i, pos - p->bounds[k], t, int32_t(end - i), k, 0});
            i = end;
        }
    }
}

}  // namespace

extern "C" int dbuf_plan(const dbuf_tensor_spec *specs, int32_t n, int32_t m,
                         const int32_t *local_units, int64_t align_elems, dbuf_plan_t **out) {
    if (!out) return DBUF_EINVAL;
    *out = nullptr;
    int rc = validate(specs, n, m, local_units, align_elems);
    if (rc != DBUF_OK) return rc;
    dbuf_plan_t *p = new (std::nothrow) dbuf_plan_t();
    if (!p) return DBUF_ENOMEM;
    try {
        p->n = n;
        p->m = m;
        p->align = align_elems;
        p->even = (local_units == nullptr);
        p->specs.assign(specs, specs + n);
        p->units.assign(m, 1);
        if (local_units) std::copy(local_units, local_units + m, p->units.begin());

        std::vector<int64_t> c(m + 1, 0);
        int64_t umax = 0;
        for (int k = 0; k < m; ++k) {
            c[k + 1] = c[k] + p->units[k];
            umax = std::max<int64_t>(umax, p->units[k]);
        }
        const int64_t a = align_elems;
        std::vector<TensorGeom> ts(n);
        std::vector<std::pair<int64_t, int64_t>> thr;
        int64_t E = 0, big = 0;
        for (int32_t t = 0; t < n; ++t) {
            const dbuf_tensor_spec &s = specs[t];
            const int64_t numel = s.rows * s.cols;
            int64_t g = (s.gran_rows <= 0 || s.gran_rows >= s.rows) ? numel : s.gran_rows * s.cols;
            if (g < 1) g = 1;
            ts[t].n = numel;
            ts[t].g = g;
            ts[t].L = a / gcd64(a, g) * g;
            E += numel;
            big = std::max(big, std::min(g, numel));
            if (g < numel) thr.emplace_back((numel - 1) / 2, g);
        }
        std::sort(thr.begin(), thr.end(),
                  [](const std::pair<int64_t, int64_t> &x, const std::pair<int64_t, int64_t> &y) {
                      return x.first > y.first;
                  });
        std::vector<int64_t> rem(n + 1, 0), P(n + 1, 0);
        for (int32_t t = n - 1; t >= 0; --t) rem[t] = rem[t + 1] + ts[t].n;
        for (int32_t t = 0; t < n; ++t) P[t + 1] = P[t] + round_up(ts[t].n, a);

        int64_t lb = (E + c[m] - 1) / c[m];
        lb = std::max(lb, (big + umax - 1) / umax);
        lb = round_up(lb, a);

        p->offsets.assign(n, 0);
        std::vector<int64_t> off(n > 0 ? n : 1);
        int64_t S = lb;
        for (;;) {
            if (p->even) S = next_candidate(S, a, thr);
            Geometry geo{p->even, m, S, c.data()};
            if (feasible(ts, P, rem, a, geo)) {
                if (!place(ts, rem, a, geo, off.data())) {  // the two checks agree by construction
                    delete p;
                    return DBUF_EINVAL;
                }
                break;
            }
            S += a;
        }
        p->S = S;
        p->total = S * c[m];
        std::copy(off.begin(), off.begin() + n, p->offsets.begin());
        p->bounds.resize(m + 1);
        for (int k = 0; k <= m; ++k) p->bounds[k] = S * c[k];
        build_tables(p);
        if (p->chunks.size() > size_t(INT32_MAX) || p->tile_items.size() > size_t(INT32_MAX) ||
            p->row_items.size() > size_t(INT32_MAX) || p->pipe_items.size() > size_t(INT32_MAX) ||
            p->opt_items.size() + p->opt_plain.size() > size_t(INT32_MAX) ||
            p->pieces.size() > size_t(INT32_MAX) || p->p8_items.size() > size_t(INT32_MAX) ||
            p->big_items.size() > size_t(INT32_MAX)) {
            delete p;
            return DBUF_ERANGE;
        }
    } catch (const std::bad_alloc &) {
        delete p;
        return DBUF_ENOMEM;
    }
    *out = p;
    return DBUF_OK;
}

extern "C" int dbuf_plan_slice(const dbuf_plan_t *p, int32_t k, dbuf_plan_t **out) {
    if (!out) return DBUF_EINVAL;
    *out = nullptr;
    if (!p || p->slice_k >= 0 || k < 0 || k >= p->m) return DBUF_EINVAL;
    dbuf_plan_t *s = new (std::nothrow) dbuf_plan_t();
    if (!s) return DBUF_ENOMEM;
    try {
        const int32_t n = p->n;
        const int64_t B0 = p->bounds[k], B1 = p->bounds[k + 1], len = B1 - B0;
        s->n = n;
        s->m = 1;
        s->align = p->align;
        s->even = true;
        s->units.assign(1, 1);
        s->S = len;
        s->total = len;
        s->bounds = {0, len};
        s->slice_k = k;
        s->slice_base = B0;
        s->specs.resize(n);
        s->offsets.assign(n, 0);
        s->src_offsets.assign(n, 0);
        int64_t scale_base = 0;
        for (int32_t t = 0; t < n; ++t) {
            const dbuf_tensor_spec &ps = p->specs[t];
            const int64_t l = p->offsets[t], nt = ps.rows * ps.cols;
            const int64_t lo = std::max(l, B0), hi = std::min(l + nt, B1);
            dbuf_tensor_spec ss = ps;
            ss.gran_rows = 0;
            if (hi > lo) {
                const int64_t e0 = lo - l, pl = hi - lo;
                s->offsets[t] = lo - B0;
                s->src_offsets[t] = e0;
                if (ps.quant != DBUF_QUANT_NONE) {
                    // shard cuts fall on whole units, and a quantised tensor's unit is a
                    // whole number of block rows: the piece is rows [r0, r0 + pr)
                    const int64_t qr =
                        ps.qblock_rows > 0 ? ps.qblock_rows : std::max<int64_t>(ps.rows, 1);
                    const int64_t blk_row = qr * ps.cols;
                    if (e0 % blk_row != 0 || (hi != l + nt && pl % blk_row != 0)) {
                        delete s;
                        return DBUF_EINVAL;
                    }
                    ss.rows = pl / ps.cols;
                    ss.qblock_rows = int32_t(qr);
                } else {
                    ss.rows = pl;
                    ss.cols = 1;
                }
            } else {
                s->offsets[t] = std::min(std::max<int64_t>(l - B0, 0), len);
                s->src_offsets[t] = l + nt <= B0 ? nt : 0;
                ss.rows = 0;
                if (ps.quant == DBUF_QUANT_NONE) ss.cols = 1;
            }
            s->specs[t] = ss;
            // global block scales that lie before the slice
            if (ps.quant != DBUF_QUANT_NONE && nt > 0) {
                const int64_t qr =
                    ps.qblock_rows > 0 ? ps.qblock_rows : std::max<int64_t>(ps.rows, 1);
                const int64_t qc =
                    ps.qblock_cols > 0 ? ps.qblock_cols : std::max<int64_t>(ps.cols, 1);
                const int64_t nbc = (ps.cols + qc - 1) / qc, nbr = (ps.rows + qr - 1) / qr;
                if (l + nt <= B0) scale_base += nbr * nbc;
                else if (l < B0) scale_base += (B0 - l) / (qr * ps.cols) * nbc;
            }
        }
        s->scale_base = scale_base;
        build_tables(s);
        if (s->chunks.size() > size_t(INT32_MAX) || s->pieces.size() > size_t(INT32_MAX) ||
            s->pipe_items.size() > size_t(INT32_MAX) || s->p8_items.size() > size_t(INT32_MAX) ||
            s->big_items.size() > size_t(INT32_MAX) ||
            s->opt_items.size() + s->opt_plain.size() > size_t(INT32_MAX)) {
            delete s;
            return DBUF_ERANGE;
        }
    } catch (const std::bad_alloc &) {
        delete s;
        return DBUF_ENOMEM;
    }
    *out = s;
    return DBUF_OK;
}

extern "C" int dbuf_plan_slice_info(const dbuf_plan_t *s, int32_t *k, int64_t *global_offset,
                                    int64_t *src_offsets, int64_t *numels, int64_t *scale_base) {
    if (!s || s->slice_k < 0) return DBUF_EINVAL;
    if (k) *k = s->slice_k;
    if (global_offset) *global_offset = s->slice_base;
    for (int32_t t = 0; t < s->n; ++t) {
        if (src_offsets) src_offsets[t] = s->src_offsets[t];
        if (numels) numels[t] = s->tdesc[t].numel;
    }
    if (scale_base) *scale_base = s->scale_base;
    return DBUF_OK;
}

extern "C" int dbuf_plan_query(const dbuf_plan_t *p, int64_t *S, int64_t *total,
                               int64_t *offsets, int64_t *shard_bounds, int64_t *scale_offsets,
                               int64_t *n_scales) {
    if (!p) return DBUF_EINVAL;
    if (S) *S = p->S;
    if (total) *total = p->total;
    if (offsets && p->n) std::memcpy(offsets, p->offsets.data(), sizeof(int64_t) * p->n);
    if (shard_bounds) std::memcpy(shard_bounds, p->bounds.data(), sizeof(int64_t) * (p->m + 1));
    if (scale_offsets && p->n)
        std::memcpy(scale_offsets, p->scale_offsets.data(), sizeof(int64_t) * p->n);
    if (n_scales) *n_scales = p->n_scales;
    return DBUF_OK;
}

extern "C" int dbuf_order(const dbuf_tensor_spec *specs, int32_t n, int32_t kind, int32_t *perm) {
    if (n < 0 || (n > 0 && (!specs || !perm))) return DBUF_EINVAL;
    if (kind != DBUF_ORDER_DEFAULT && kind != DBUF_ORDER_BLOCK && kind != DBUF_ORDER_SHAPE)
        return DBUF_EINVAL;
    std::vector<int32_t> idx(n);
    for (int32_t t = 0; t < n; ++t) idx[t] = t;
    auto unit = [&](int32_t t) {
        const dbuf_tensor_spec &s = specs[t];
        const int64_t numel = s.rows * s.cols;
        const int64_t g = (s.gran_rows <= 0 || s.gran_rows >= s.rows) ? numel : s.gran_rows * s.cols;
        return std::max<int64_t>(g, 1);
    };
    if (kind == DBUF_ORDER_BLOCK)
        std::stable_sort(idx.begin(), idx.end(),
                         [&](int32_t a, int32_t b) { return unit(a) > unit(b); });
    else if (kind == DBUF_ORDER_SHAPE)
        std::stable_sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) {
            if (specs[a].rows != specs[b].rows) return specs[a].rows > specs[b].rows;
            return specs[a].cols > specs[b].cols;
        });
    std::copy(idx.begin(), idx.end(), perm);
    return DBUF_OK;
}

extern "C" int dbuf_plan_state_offsets(const dbuf_plan_t *p, int64_t *state_offsets,
                                       int64_t *n_state) {
    if (!p) return DBUF_EINVAL;
    if (state_offsets && p->n)
        std::memcpy(state_offsets, p->state_offsets.data(), sizeof(int64_t) * p->n);
    if (n_state) *n_state = p->n_state;
    return DBUF_OK;
}

extern "C" const char *dbuf_strerror(int code) {
    switch (code) {
        case DBUF_OK: return "ok";
        case DBUF_EINVAL: return "invalid argument";
        case DBUF_ENOMEM: return "out of memory";
        case DBUF_ECUDA: return "CUDA error";
        case DBUF_ENOTUPLOADED: return "plan not uploaded to the device";
        case DBUF_ETIMEOUT: return "device-side wait timed out";
        case DBUF_EDEVICE: return "current device differs from the plan's device";
        case DBUF_ERANGE: return "size out of range";
        default: return "unknown error";
    }
}

extern "C" size_t dbuf_workspace_bytes(const dbuf_plan_t *p, int32_t op) {
    if (!p) return 0;
    if (op == DBUF_OP_NORM_NONFINITE) return dbuf::norm_workspace_bytes(p);
    return 0;
}
