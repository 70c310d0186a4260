// Host tile planner of the GDPA library.
//
// The GDPA page ("범용 내적 어텐션(GDPA): 실제 추천 시스템 학습 부하를 위한
// 커널 최적화", aitrends.kr, "섹션별 상세", the paragraph on jagged inputs and
// the zigzag-scheduling diagram) has the CPU compute the valid tiles of a
// jagged batch ahead of the launch and hand them to the SMs in a zigzag
// pattern after sorting, in place of round robin, to even out SM load.
//
// Rules (the page gives only the idea; these are the library's definitions):
//  * forward tile  = (sample b, head h, query tile m); its key blocks are the
//    hull of the valid keys of its rows (no mask: all keys; causal window W:
//    [m*BM - W + 1, min((m+1)*BM, Lq))), clipped to [0, Lkv).  An empty hull
//    gives a zero tile (kb0 = kb1 = 0) whose rows the kernel writes as zeros.
//  * backward unit = (b, h, key block j); its query tiles are the hull of the
//    queries that see a key of the block.  A sample whose query tiles are
//    reached by more than one key block gets its dQ by atomic adds.
//  * key split (max_kv_blocks_per_tile = k > 0): a forward tile's key blocks
//    are cut into chunks of at most k, each its own tile; automatic choice
//    (k = GDPA_KV_SPLIT_AUTO): chunks of 2 when some query tile reaches 8 or
//    more key blocks, else no split (measured on the pooling workload,
//    32 queries against up to 8192 keys per sample: 2-block chunks were the
//    fastest at 16, 64 and 1024 samples).
//  * cost = blocks on the inner loop; zigzag = stable sort by cost,
//    descending, then snake dealing over the S SMs; round robin = tile r to
//    SM r % S in enumeration order.  Timed zigzag deals the same way but
//    costs backward units with the integer time model of include/gdpa.h
//    (GDPA_SCHED_ZIGZAG_TIMED).
#include <algorithm>
#include <numeric>

#include "gdpa_internal.h"

namespace gdpa {
namespace {

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t up(int64_t a, int64_t m) { return cdiv(a, m) * m; }

// The time model of GDPA_SCHED_ZIGZAG_TIMED (units of 50 ns).
// Backward unit: nkv keys, query tiles [m0, m1) of a sample with lq queries.
int64_t bwd_time_cost(int64_t nkv, int64_t m0, int64_t m1, int64_t lq) {
    if (m1 <= m0) return 1;
    const int64_t k16 = up(nkv, 16);
    int64_t c = 36 + 22 * k16 / 128;
    for (int64_t m = m0; m < m1; ++m)
        c += 40 + 34 * up(std::min<int64_t>(kBM, lq - m * kBM), 32) / 128 + 24 * k16 / 128;
    return c;
}

struct Item {
    int32_t f[6];  // forward: b h m kb0 kb1 -; backward: b h j m0 m1 flags
    int64_t cost;
};

// Deal items to S queues; returns the SM of each item in dealing order.
void deal(const std::vector<Item>& items, int S, int sched, std::vector<int64_t>& order,
          std::vector<int32_t>& sm) {
    const int64_t n = (int64_t)items.size();
    order.resize(n);
    std::iota(order.begin(), order.end(), 0);
    const bool zz = sched == GDPA_SCHED_ZIGZAG || sched == GDPA_SCHED_ZIGZAG_TIMED;
    if (zz) {
        // stable sort by cost, descending: a counting sort when the costs
        // span a small range (they count blocks or tiles), else a merge sort
        int64_t cmax = 0;
        for (const Item& it : items) cmax = std::max(cmax, it.cost);
        if (cmax < (int64_t)1 << 16) {
            std::vector<int64_t> start(cmax + 2, 0);
            for (const Item& it : items) start[cmax - it.cost + 1]++;
            for (int64_t c = 0; c <= cmax; ++c) start[c + 1] += start[c];
            for (int64_t i = 0; i < n; ++i) order[start[cmax - items[i].cost]++] = i;
        } else {
            std::stable_sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
                return items[a].cost > items[b].cost;
            });
        }
    }
    sm.resize(n);
    int32_t col = 0;
    bool odd = false;   // odd dealing round: the snake runs back
    for (int64_t r = 0; r < n; ++r) {
        sm[r] = (zz && odd) ? S - 1 - col : col;
        if (++col == S) {
            col = 0;
            odd = !odd;
        }
    }
}

// Group dealt items by SM (stable within an SM), emit export rows and call
// record(q, item) for the items at queue positions q = 0, 1, 2, ... in turn.
template <int W, typename Record>
void emit(const std::vector<Item>& items, int S, int sched, std::vector<int32_t>& rows,
          std::vector<int32_t>& seg, Record record) {
    std::vector<int64_t> queue_order;
    std::vector<int64_t> order;
    std::vector<int32_t> sm;
    deal(items, S, sched, order, sm);
    std::vector<int64_t> count(S + 1, 0);
    for (int64_t r = 0; r < (int64_t)order.size(); ++r) count[sm[r] + 1]++;
    for (int s = 0; s < S; ++s) count[s + 1] += count[s];
    seg.assign(count.begin(), count.end());
    queue_order.assign(order.size(), 0);
    std::vector<int64_t> fill(count.begin(), count.end() - 1);
    for (int64_t r = 0; r < (int64_t)order.size(); ++r) queue_order[fill[sm[r]]++] = order[r];
    // queue positions run 0, 1, 2, ... in this loop: append, no zero fill
    const int64_t n = (int64_t)queue_order.size();
    rows.clear();
    rows.reserve(n * W);
    for (int s = 0; s < S; ++s) {
        for (int64_t q = count[s]; q < count[s + 1]; ++q) {
            if (q + 8 < n) __builtin_prefetch(&items[queue_order[q + 8]]);
            const Item& it = items[queue_order[q]];
            for (int c = 0; c < W - 1; ++c) rows.push_back(it.f[c]);
            rows.push_back(s);
            record(q, it);
        }
    }
}

}  // namespace

gdpa_status build_plan_host(Plan& p, const int32_t* q_off, const int32_t* kv_off) {
    const int B = p.B, H = p.H, S = p.S;
    if (q_off[0] != 0 || kv_off[0] != 0) return GDPA_ERR_INVALID_ARG;
    for (int b = 0; b < B; ++b)
        if (q_off[b + 1] < q_off[b] || kv_off[b + 1] < kv_off[b]) return GDPA_ERR_INVALID_ARG;
    p.Tq = q_off[B];
    p.Tkv = kv_off[B];
    p.max_lq = 0;
    for (int b = 0; b < B; ++b) p.max_lq = std::max<int64_t>(p.max_lq, q_off[b + 1] - q_off[b]);
    const bool win = p.mask == GDPA_MASK_CAUSAL_WINDOW;
    const bool timed = p.sched == GDPA_SCHED_ZIGZAG_TIMED;
    const int64_t W = p.window;
    // key-block hull of query tile m of sample b (empty: k0 = k1 = 0)
    auto kv_hull = [&](int b, int64_t m, int64_t& k0, int64_t& k1) {
        const int64_t lq = q_off[b + 1] - q_off[b], lkv = kv_off[b + 1] - kv_off[b];
        const int64_t r0 = m * kBM, r1 = std::min<int64_t>(r0 + kBM, lq);
        int64_t lo = 0, hi = lkv;
        if (win) {
            lo = std::max<int64_t>(0, r0 - W + 1);
            hi = std::min<int64_t>(lkv, r1);
        }
        k0 = k1 = 0;
        if (lo < hi) {
            k0 = lo / kBN;
            k1 = cdiv(hi, kBN);
        }
    };
    if (p.max_kvb == GDPA_KV_SPLIT_AUTO) {
        int64_t widest = 0;
        for (int b = 0; b < B; ++b)
            for (int64_t m = 0; m < cdiv(q_off[b + 1] - q_off[b], kBM); ++m) {
                int64_t k0, k1;
                kv_hull(b, m, k0, k1);
                widest = std::max(widest, k1 - k0);
            }
        p.max_kvb = widest >= 8 ? 2 : 0;
    }

    // forward tiles, enumerated b -> h -> m (-> chunk)
    std::vector<Item> ft;
    {
        // an upper bound of the tile count (key chunks counted over the
        // sample's whole key range), so that the vectors never reallocate
        int64_t bound = 0;
        for (int b = 0; b < B; ++b) {
            const int64_t nkb = cdiv(kv_off[b + 1] - kv_off[b], kBN);
            const int64_t chunks = p.max_kvb > 0 ? std::max<int64_t>(1, cdiv(nkb, p.max_kvb)) : 1;
            bound += H * cdiv(q_off[b + 1] - q_off[b], kBM) * chunks;
        }
        ft.reserve(bound);
    }
    p.max_fwd_kvb = 0;
    p.fwd_split = 0;
    for (int b = 0; b < B; ++b) {
        const int64_t lq = q_off[b + 1] - q_off[b];
        for (int h = 0; h < H; ++h) {
            for (int64_t m = 0; m < cdiv(lq, kBM); ++m) {
                int64_t k0, k1;
                kv_hull(b, m, k0, k1);
                const int64_t step = (p.max_kvb > 0 && k1 > k0) ? p.max_kvb : std::max<int64_t>(1, k1 - k0);
                int64_t s = k0;
                do {
                    const int64_t e = std::min(k1, s + step);
                    ft.push_back(Item{{b, h, (int32_t)m, (int32_t)s, (int32_t)e, 0}, e - s});
                    p.max_fwd_kvb = std::max<int64_t>(p.max_fwd_kvb, e - s);
                    if (e - s < k1 - k0) p.fwd_split = 1;
                    s = e;
                } while (s < k1);
            }
        }
    }

    // backward units, enumerated b -> h -> j
    std::vector<Item> bu;
    {
        int64_t units = 0;
        for (int b = 0; b < B; ++b) units += H * cdiv(kv_off[b + 1] - kv_off[b], kBN);
        bu.reserve(units);
    }
    p.zero_dq = 0;
    for (int b = 0; b < B; ++b) {
        const int64_t lq = q_off[b + 1] - q_off[b], lkv = kv_off[b + 1] - kv_off[b];
        const int64_t nkb = cdiv(lkv, kBN), nm = cdiv(lq, kBM);
        std::vector<int64_t> m0s(nkb), m1s(nkb);
        for (int64_t j = 0; j < nkb; ++j) {
            const int64_t c0 = j * kBN, c1 = std::min<int64_t>(c0 + kBN, lkv);
            int64_t lo = 0, hi = lq;
            if (win) {
                lo = c0;
                hi = std::min<int64_t>(lq, c1 - 1 + W);
            }
            m0s[j] = lo < hi ? lo / kBM : 0;
            m1s[j] = lo < hi ? cdiv(hi, kBM) : 0;
        }
        // query-tile coverage count: atomic dQ if any tile is reached twice,
        // clearing needed if any tile is never reached
        std::vector<int32_t> cover(nm, 0);
        for (int64_t j = 0; j < nkb; ++j)
            for (int64_t m = m0s[j]; m < m1s[j]; ++m) cover[m]++;
        bool atomic = false, hole = false;
        for (int64_t m = 0; m < nm; ++m) {
            atomic |= cover[m] > 1;
            hole |= cover[m] == 0;
        }
        if (atomic || hole) p.zero_dq = 1;
        const int32_t flags = atomic ? kUnitAtomicDQ : 0;
        for (int h = 0; h < H; ++h) {
            for (int64_t j = 0; j < nkb; ++j) {
                const int64_t cost =
                    timed ? bwd_time_cost(std::min<int64_t>(kBN, lkv - j * kBN), m0s[j], m1s[j], lq)
                          : m1s[j] - m0s[j];
                bu.push_back(Item{{b, h, (int32_t)j, (int32_t)m0s[j], (int32_t)m1s[j], flags},
                                  cost});
            }
        }
    }

    // kernel-layout records in queue order (uploaded by the ABI layer),
    // written as the items are grouped by SM
    std::vector<FwdTile> fdev;
    fdev.reserve(ft.size());
    emit<6>(ft, S, p.sched, p.fwd_export, p.fwd_seg, [&](int64_t, const Item& it) {
        const int b = it.f[0];
        const int64_t lq = q_off[b + 1] - q_off[b], r0 = (int64_t)it.f[2] * kBM;
        FwdTile& t = fdev.emplace_back();
        t.qt0 = (int32_t)(q_off[b] + r0);
        t.nq = (int32_t)(std::min<int64_t>(r0 + kBM, lq) - r0);
        t.kvt0 = kv_off[b];
        t.lkv = kv_off[b + 1] - kv_off[b];
        t.h = it.f[1];
        t.kb0 = it.f[3];
        t.kb1 = it.f[4];
        t.i0 = (int32_t)r0;
    });
    p.n_fwd = (int64_t)ft.size();
    std::vector<BwdUnit> bdev;
    bdev.reserve(bu.size());
    emit<7>(bu, S, p.sched, p.bwd_export, p.bwd_seg, [&](int64_t, const Item& it) {
        const int b = it.f[0];
        const int64_t lkv = kv_off[b + 1] - kv_off[b], c0 = (int64_t)it.f[2] * kBN;
        BwdUnit& u = bdev.emplace_back();
        u.kvt0 = (int32_t)(kv_off[b] + c0);
        u.nkv = (int32_t)(std::min<int64_t>(c0 + kBN, lkv) - c0);
        u.qt0 = q_off[b];
        u.lq = q_off[b + 1] - q_off[b];
        u.hf = it.f[1] | (it.f[5] << 16);
        u.m0 = it.f[3];
        u.m1 = it.f[4];
        u.c0 = (int32_t)c0;
    });
    p.n_bwd = (int64_t)bu.size();
    p.fwd_dev_host.swap(fdev);
    p.bwd_dev_host.swap(bdev);
    return GDPA_OK;
}


// ---------------------------------------------------------------- sharding

extern "C" gdpa_status gdpa_shard_batch(const int32_t* q_off, const int32_t* kv_off, int B, int H,
                                        gdpa_mask mask, int window, int num_ranks,
                                        int32_t* rank_out, int64_t* work_out) {
    if (!q_off || !kv_off || B < 0 || H < 1 || num_ranks < 1 || (B > 0 && !rank_out))
        return GDPA_ERR_INVALID_ARG;
    if (mask != GDPA_MASK_NONE && mask != GDPA_MASK_CAUSAL_WINDOW) return GDPA_ERR_INVALID_ARG;
    if (mask == GDPA_MASK_CAUSAL_WINDOW && window < 1) return GDPA_ERR_INVALID_ARG;
    if (q_off[0] != 0 || kv_off[0] != 0) return GDPA_ERR_INVALID_ARG;
    for (int b = 0; b < B; ++b)
        if (q_off[b + 1] < q_off[b] || kv_off[b + 1] < kv_off[b]) return GDPA_ERR_INVALID_ARG;
    const bool win = mask == GDPA_MASK_CAUSAL_WINDOW;
    // a sample's work: H x the key blocks of its query tiles (the forward
    // tile cost of gdpa_plan_create, summed over the sample)
    std::vector<Item> items(B);
    for (int b = 0; b < B; ++b) {
        const int64_t lq = q_off[b + 1] - q_off[b], lkv = kv_off[b + 1] - kv_off[b];
        int64_t w = 0;
        for (int64_t m = 0; m < cdiv(lq, kBM); ++m) {
            const int64_t r0 = m * kBM, r1 = std::min<int64_t>(r0 + kBM, lq);
            int64_t lo = 0, hi = lkv;
            if (win) {
                lo = std::max<int64_t>(0, r0 - window + 1);
                hi = std::min<int64_t>(lkv, r1);
            }
            if (lo < hi) w += cdiv(hi, kBN) - lo / kBN;
        }
        items[b] = Item{{b, 0, 0, 0, 0, 0}, w * H};
    }
    std::vector<int64_t> order;
    std::vector<int32_t> rank;
    deal(items, num_ranks, GDPA_SCHED_ZIGZAG, order, rank);
    if (work_out)
        for (int r = 0; r < num_ranks; ++r) work_out[r] = 0;
    for (int64_t k = 0; k < (int64_t)order.size(); ++k) {
        rank_out[order[k]] = rank[k];
        if (work_out) work_out[rank[k]] += items[order[k]].cost;
    }
    return GDPA_OK;
}

}  // namespace gdpa
