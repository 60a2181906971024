// Explicit-state checker of mbarrier protocols (host code only).
//
// The CUTLASS Task Scheduling pages check a captured schedule statically for
// deadlocks and races before lowering it ("Introduction", the verifier behind
// TaskManager.print_and_verify).  tile_scheduling_gb300/protocol.py restates
// this library's GEMM role loops as small programs over mbarriers and buffers;
// this engine explores every interleaving of those programs and of the
// asynchronous units they drive, depth first, keeping a 64-bit hash of each
// visited state (hash compaction).
//
// Program model.  Barriers start in phase 0 with `expected` pending arrivals
// and no transaction bytes.  A phase completes when pending arrivals and
// transaction bytes both reach zero (complete-tx may run ahead of the matching
// expect-tx and drive the count below zero).  A wait on parity P passes while
// the number of completed phases has the other parity.  Op records are 8
// int32 wide:
//   WAIT   bar parity            ARRIVE bar tx_bytes (expect-tx, then arrive)
//   TMA    buf tag bar bytes     -> async: buf := tag, then complete-tx(bar)
//   MMA    sbuf0 sbuf1 acc tag sbuf2 sbuf3
//                                -> in-order queue: the (up to four) sbufs must
//                                   hold tag; a tag with k-block > 0 must find
//                                   tag - 1 in acc
//   COMMIT bar0 bar1             -> in-order queue: one arrival on each bar
//   TREAD  buf tag               buf must hold tag
//   CREQ   slot0 slot1 seq bar0 bar1 bytes  -> async: slots := seq, complete-tx
//   CREAD  buf seq               buf must hold seq
//   GWRITE buf tag               -> async: buf := tag (a global-memory store,
//                                   visible to other roles once it lands)
//   FENCE                        blocks while a GWRITE of this role is in flight
//   TICKET ctr last buf0 nbufs tag0 rearm
//                                fetch-and-add on counter ctr; the role that
//                                draws `last` re-arms the counter to 0 (if rearm)
//                                and reads bufs buf0 .. buf0 + nbufs - 1, which
//                                must hold tag0, tag0 + 1, ...
//   TREADB buf limit             buf must hold a tag below limit (a read whose
//                                data is discarded: only a later writer races it)
// (negative operands mean "none"; tags are unit * 1024 + k-block.)  A role step
// runs one wait, fence, arrive or ticket plus the ops after it that only enqueue
// work or, after a wait, only check a buffer: their effects become visible
// later, through the queue or the async completions, which are explored
// separately.  Counters start at 0; when every role has finished, each must be
// back at 0 and have been drawn `last` exactly its expected number of times.
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "common.h"

namespace ts {
namespace {

enum : int32_t {
    OP_WAIT = 0,
    OP_ARRIVE,
    OP_TMA,
    OP_MMA,
    OP_COMMIT,
    OP_TREAD,
    OP_CREQ,
    OP_CREAD,
    OP_GWRITE,
    OP_FENCE,
    OP_TICKET,
    OP_TREADB
};
constexpr int kRec = 8;
constexpr int kMaxQueue = 32;
constexpr int kMaxAsync = 32;

struct Model {
    int nbars, nbufs, nroles, nctrs;
    const int32_t *expected, *group, *off, *ops, *ctr_expected;
    std::vector<std::string> role_name, bar_name, buf_name;
    // state layout offsets
    int o_pc, o_bar, o_buf, o_mq, o_asy, o_ctr, len;
};

struct Checker {
    const Model &m;
    std::vector<uint64_t> table;  // open addressing, load factor at most one half; grows by doubling
    uint64_t mask;
    int64_t states = 0, max_states;
    std::string msg;

    Checker(const Model &mm, int64_t maxs) : m(mm), max_states(maxs) {
        table.assign(uint64_t(1) << 16, 0);
        mask = table.size() - 1;
    }

    // Hash of the live words of a state: the unused tails of the tcgen05 queue
    // and of the in-flight list always hold -1, so they are left out.  Four
    // independent lanes (words 4j, 4j + 1, 4j + 2 and 4j + 3 of each part) keep
    // the multiplies from forming one long dependency chain.
    uint64_t hash(const int32_t *s) const {
        uint64_t h[4] = {0x9E3779B97F4A7C15ull, 0xC2B2AE3D27D4EB4Full, 0x165667B19E3779F9ull, 0x27D4EB2F165667C5ull};
        auto step = [](uint64_t &x, int32_t v) {
            x = (x ^ static_cast<uint32_t>(v)) * 0x100000001B3ull;
            x ^= x >> 29;
        };
        auto mix = [&](const int32_t *p, int n) {
            int k = 0;
            for (; k + 3 < n; k += 4) {
                step(h[0], p[k]);
                step(h[1], p[k + 1]);
                step(h[2], p[k + 2]);
                step(h[3], p[k + 3]);
            }
            for (int j = 0; k < n; ++k, ++j) step(h[j], p[k]);
            step(h[3], n);
        };
        mix(s, m.o_mq + 1 + s[m.o_mq]);  // pcs, barriers, buffers, the queue's length and entries
        mix(s + m.o_asy, 1 + s[m.o_asy]);
        mix(s + m.o_ctr, m.len - m.o_ctr);
        uint64_t x = h[0];
        for (int j = 1; j < 4; ++j) {
            x ^= (h[j] ^ (h[j] >> 31)) * (0x9E3779B97F4A7C15ull + 2 * static_cast<uint64_t>(j));
            x ^= x >> 32;
        }
        return x ? x : 1;
    }

    void grow() {
        std::vector<uint64_t> old(table.size() * 2, 0);
        old.swap(table);
        mask = table.size() - 1;
        for (uint64_t h : old) {
            if (!h) continue;
            uint64_t i = h & mask;
            while (table[i]) i = (i + 1) & mask;
            table[i] = h;
        }
    }

    void prefetch(uint64_t h) const { __builtin_prefetch(&table[h & mask]); }

    bool insert(uint64_t h) {  // true if new
        for (uint64_t i = h & mask;; i = (i + 1) & mask) {
            if (table[i] == h) return false;
            if (table[i] == 0) {
                table[i] = h;
                ++states;
                if (2 * static_cast<uint64_t>(states) > table.size()) grow();
                return true;
            }
        }
    }

    void canon(int32_t *s) const {
        // copies in flight form a set: keep them sorted
        std::sort(s + m.o_asy + 1, s + m.o_asy + 1 + s[m.o_asy]);
        // roles of one symmetry group run identical programs: keep their pcs sorted
        for (int i = 0; i < m.nroles; ++i) {
            if (m.group[i] < 0) continue;
            for (int j = i + 1; j < m.nroles; ++j)
                if (m.group[j] == m.group[i] && s[m.o_pc + j] < s[m.o_pc + i]) std::swap(s[m.o_pc + i], s[m.o_pc + j]);
        }
    }

    const int32_t *op(int idx) const { return m.ops + static_cast<int64_t>(idx) * kRec; }

    // returns false on over-arrival
    bool arrive(int32_t *s, int b, int tx) const {
        int32_t *bs = s + m.o_bar + 3 * b;
        bs[1] -= 1;
        bs[2] += tx;
        if (bs[1] < 0) return false;
        if (bs[1] == 0 && bs[2] == 0) {
            bs[0] += 1;
            bs[1] = m.expected[b];
        }
        return true;
    }
    void complete_tx(int32_t *s, int b, int bytes) const {
        int32_t *bs = s + m.o_bar + 3 * b;
        bs[2] -= bytes;
        if (bs[1] == 0 && bs[2] == 0) {
            bs[0] += 1;
            bs[1] = m.expected[b];
        }
    }
    static bool push_list(int32_t *s, int o, int cap, int v) {
        int32_t &n = s[o];
        if (n >= cap) return false;
        s[o + 1 + n] = v;
        ++n;
        return true;
    }

    bool violation(const std::string &what) {
        msg = what;
        return false;
    }

    // True if role i's next op cannot run in state s (a wait on an incomplete
    // phase, or a fence behind one of its own stores in flight).
    bool blocked_at(const int32_t *s, int i, const int32_t *o) const {
        if (o[0] == OP_WAIT) return s[m.o_bar + 3 * o[1]] % 2 == o[2];
        if (o[0] == OP_FENCE) {
            for (int k = 0; k < s[m.o_asy]; ++k) {
                const int idx = s[m.o_asy + 1 + k];
                if (idx >= m.off[i] && idx < m.off[i + 1]) return true;
            }
        }
        return false;
    }

    // Successors of `s`, appended to `out` (m.len words each); false if a
    // violation was found (msg set).
    bool expand(const int32_t *s, std::vector<int32_t> &out, bool &any) {
        any = false;
        std::pair<int, int> tried[64];  // (group, pc) of the symmetric roles tried
        int ntried = 0;
        std::vector<std::pair<int, int>> tried_more;
        auto start = [&]() -> int32_t * {  // a new successor, a copy of s
            const size_t base = out.size();
            out.resize(base + m.len);
            std::memcpy(&out[base], s, sizeof(int32_t) * m.len);
            return &out[base];
        };
        for (int i = 0; i < m.nroles; ++i) {
            int pc = s[m.o_pc + i];
            const int end = m.off[i + 1] - m.off[i];
            if (pc >= end) continue;
            if (m.group[i] >= 0) {
                std::pair<int, int> key(m.group[i], pc);
                if (std::find(tried, tried + ntried, key) != tried + ntried ||
                    std::find(tried_more.begin(), tried_more.end(), key) != tried_more.end())
                    continue;
                if (ntried < 64)
                    tried[ntried++] = key;
                else
                    tried_more.push_back(key);
            }
            if (blocked_at(s, i, op(m.off[i] + pc))) continue;  // blocked at its first op
            int32_t *t = start();
            bool first = true, arrived = false;
            while (pc < end) {
                const int32_t *o = op(m.off[i] + pc);
                const int kind = o[0];
                if ((kind == OP_WAIT || kind == OP_ARRIVE || kind == OP_FENCE || kind == OP_TICKET) && !first) break;
                if ((kind == OP_TREAD || kind == OP_CREAD || kind == OP_TREADB) && arrived) break;
                if (kind == OP_WAIT) {
                    if (t[m.o_bar + 3 * o[1]] % 2 == o[2]) break;
                } else if (kind == OP_FENCE) {
                    if (blocked_at(t, i, o)) break;
                } else if (kind == OP_TICKET) {
                    const int c = o[1];
                    const int drawn = t[m.o_ctr + 2 * c];
                    t[m.o_ctr + 2 * c] = drawn + 1;
                    if (drawn == o[2]) {
                        if (o[6]) t[m.o_ctr + 2 * c] = 0;
                        t[m.o_ctr + 2 * c + 1] += 1;
                        for (int k = 0; k < o[4]; ++k) {
                            if (t[m.o_buf + o[3] + k] != o[5] + k) {
                                char b[256];
                                snprintf(b, sizeof b, "%s: reduction read %s holding tag %d, expected %d",
                                         m.role_name[i].c_str(), m.buf_name[o[3] + k].c_str(),
                                         t[m.o_buf + o[3] + k], o[5] + k);
                                return violation(b);
                            }
                        }
                    }
                    arrived = true;
                } else if (kind == OP_GWRITE) {
                    if (!push_list(t, m.o_asy, kMaxAsync, m.off[i] + pc)) return violation("too many copies in flight");
                } else if (kind == OP_TREADB) {
                    if (t[m.o_buf + o[1]] >= o[2]) {
                        char b[256];
                        snprintf(b, sizeof b, "%s: read of %s found tag %d, written after the read began",
                                 m.role_name[i].c_str(), m.buf_name[o[1]].c_str(), t[m.o_buf + o[1]]);
                        return violation(b);
                    }
                } else if (kind == OP_ARRIVE) {
                    if (!arrive(t, o[1], o[2]))
                        return violation(m.role_name[i] + ": more arrivals than " + m.bar_name[o[1]] +
                                         " expects in a phase");
                    arrived = true;
                } else if (kind == OP_TMA || kind == OP_CREQ) {
                    if (!push_list(t, m.o_asy, kMaxAsync, m.off[i] + pc)) return violation("too many copies in flight");
                } else if (kind == OP_MMA || kind == OP_COMMIT) {
                    if (!push_list(t, m.o_mq, kMaxQueue, m.off[i] + pc)) return violation("tcgen05 queue too deep");
                } else if (kind == OP_TREAD) {
                    if (t[m.o_buf + o[1]] != o[2]) {
                        char b[256];
                        snprintf(b, sizeof b, "%s: read of %s found tag %d, expected the finished tile %d",
                                 m.role_name[i].c_str(), m.buf_name[o[1]].c_str(), t[m.o_buf + o[1]], o[2]);
                        return violation(b);
                    }
                } else if (kind == OP_CREAD) {
                    if (t[m.o_buf + o[1]] != o[2]) {
                        char b[256];
                        snprintf(b, sizeof b, "%s: %s holds response %d, expected response %d",
                                 m.role_name[i].c_str(), m.buf_name[o[1]].c_str(), t[m.o_buf + o[1]], o[2]);
                        return violation(b);
                    }
                }
                ++pc;
                first = false;
            }
            t[m.o_pc + i] = pc;
            any = true;
        }
        // asynchronous copies and CLC responses complete in any order
        const int na = s[m.o_asy];
        for (int k = 0; k < na; ++k) {
            const int idx = s[m.o_asy + 1 + k];
            bool dup = false;
            for (int j = 0; j < k; ++j) dup |= s[m.o_asy + 1 + j] == idx;
            if (dup) continue;
            int32_t *t = start();
            // remove entry k
            for (int j = k; j < na - 1; ++j) t[m.o_asy + 1 + j] = t[m.o_asy + 2 + j];
            t[m.o_asy + na] = -1;
            t[m.o_asy] = na - 1;
            const int32_t *o = op(idx);
            if (o[0] == OP_GWRITE) {
                t[m.o_buf + o[1]] = o[2];
            } else if (o[0] == OP_TMA) {
                const int nq = s[m.o_mq];
                for (int q = 0; q < nq; ++q) {
                    const int32_t *mo = op(s[m.o_mq + 1 + q]);
                    if (mo[0] == OP_MMA && (mo[1] == o[1] || mo[2] == o[1] || mo[5] == o[1] || mo[6] == o[1])) {
                        char b[256];
                        snprintf(b, sizeof b, "copy of tag %d overwrote %s before the queued MMA of tag %d read it",
                                 o[2], m.buf_name[o[1]].c_str(), mo[4]);
                        return violation(b);
                    }
                }
                t[m.o_buf + o[1]] = o[2];
                complete_tx(t, o[3], o[4]);
            } else {
                for (int j = 1; j <= 2; ++j)
                    if (o[j] >= 0) t[m.o_buf + o[j]] = o[3];
                for (int j = 4; j <= 5; ++j)
                    if (o[j] >= 0) complete_tx(t, o[j], o[6]);
            }
            any = true;
        }
        // the tcgen05 queue executes in order
        const int nq = s[m.o_mq];
        if (nq > 0) {
            int32_t *t = start();
            for (int j = 0; j < nq - 1; ++j) t[m.o_mq + 1 + j] = t[m.o_mq + 2 + j];
            t[m.o_mq + nq] = -1;
            t[m.o_mq] = nq - 1;
            const int32_t *o = op(s[m.o_mq + 1]);
            if (o[0] == OP_MMA) {
                const int tag = o[4];
                for (const int j : {1, 2, 5, 6}) {
                    if (o[j] >= 0 && s[m.o_buf + o[j]] != tag) {
                        char b[256];
                        snprintf(b, sizeof b, "MMA of tag %d read %s holding tag %d", tag, m.buf_name[o[j]].c_str(),
                                 s[m.o_buf + o[j]]);
                        return violation(b);
                    }
                }
                if ((tag % 1024) > 0 && s[m.o_buf + o[3]] != tag - 1) {
                    char b[256];
                    snprintf(b, sizeof b, "MMA of tag %d accumulated onto tag %d in %s", tag, s[m.o_buf + o[3]],
                             m.buf_name[o[3]].c_str());
                    return violation(b);
                }
                t[m.o_buf + o[3]] = tag;
            } else {
                for (int j = 1; j <= 2; ++j)
                    if (o[j] >= 0 && !arrive(t, o[j], 0))
                        return violation("commit: more arrivals than " + m.bar_name[o[j]] + " expects in a phase");
            }
            any = true;
        }
        return true;
    }

    int run() {
        const int L = m.len;
        std::vector<int32_t> s0(L, 0);
        for (int b = 0; b < m.nbars; ++b) s0[m.o_bar + 3 * b + 1] = m.expected[b];
        for (int x = 0; x < m.nbufs; ++x) s0[m.o_buf + x] = -1;
        for (int k = 0; k < kMaxQueue; ++k) s0[m.o_mq + 1 + k] = -1;
        for (int k = 0; k < kMaxAsync; ++k) s0[m.o_asy + 1 + k] = -1;
        insert(hash(s0.data()));
        // depth-first: the stack holds states end to end, L words each
        std::vector<int32_t> stack(s0), succ, cur(L);
        std::vector<uint64_t> hs;
        while (!stack.empty()) {
            std::memcpy(cur.data(), &stack[stack.size() - L], sizeof(int32_t) * L);
            stack.resize(stack.size() - L);
            const int32_t *s = cur.data();
            succ.clear();
            bool any = false;
            if (!expand(s, succ, any)) return 1;
            if (!any) {
                std::string blocked;
                for (int i = 0; i < m.nroles; ++i) {
                    const int pc = s[m.o_pc + i];
                    if (pc >= m.off[i + 1] - m.off[i]) continue;
                    const int32_t *o = op(m.off[i] + pc);
                    if (!blocked.empty()) blocked += "; ";
                    blocked += m.role_name[i] + (o[0] == OP_WAIT ? " waiting on " + m.bar_name[o[1]] : " stuck");
                }
                if (!blocked.empty()) {
                    msg = "deadlock: " + blocked;
                    return 1;
                }
                // every role finished, nothing in flight: every counter re-armed and
                // drawn last as often as expected
                for (int c = 0; c < m.nctrs; ++c) {
                    if (s[m.o_ctr + 2 * c] != 0 || s[m.o_ctr + 2 * c + 1] != m.ctr_expected[c]) {
                        char b[256];
                        snprintf(b, sizeof b, "counter %d ends at %d after %d reductions (expected 0 after %d)", c,
                                 s[m.o_ctr + 2 * c], s[m.o_ctr + 2 * c + 1], m.ctr_expected[c]);
                        msg = b;
                        return 1;
                    }
                }
                continue;
            }
            // hash every successor first and prefetch its table slot, so the
            // (mostly cache-missing) probes of one state's successors overlap
            hs.clear();
            for (size_t at = 0; at < succ.size(); at += L) {
                canon(&succ[at]);
                hs.push_back(hash(&succ[at]));
                prefetch(hs.back());
            }
            for (size_t k = 0; k < hs.size(); ++k) {
                if (insert(hs[k])) {
                    if (states > max_states) {
                        msg = "state limit reached";
                        return 2;
                    }
                    stack.insert(stack.end(), &succ[k * L], &succ[k * L] + L);
                }
            }
        }
        msg = "no deadlock, no race";
        return 0;
    }
};

std::vector<std::string> split_lines(const char *s) {
    std::vector<std::string> v;
    std::string cur;
    for (; s && *s; ++s) {
        if (*s == '\n') {
            v.push_back(cur);
            cur.clear();
        } else {
            cur += *s;
        }
    }
    v.push_back(cur);
    return v;
}

}  // namespace
}  // namespace ts

extern "C" int32_t ts_protocol_check_ex(int32_t nbars, const int32_t *bar_expected, int32_t nbufs, int32_t nroles,
                                        const int32_t *role_group, const int32_t *role_offsets, const int32_t *ops,
                                        int32_t ncounters, const int32_t *counter_reductions, const char *names,
                                        int64_t max_states, int64_t *states_out, char *msg, int32_t msg_len) {
    using namespace ts;
    if (nbars < 0 || nbufs < 0 || nroles <= 0 || !bar_expected || !role_group || !role_offsets || !ops ||
        ncounters < 0 || (ncounters > 0 && !counter_reductions) || max_states <= 0 || !msg || msg_len <= 0)
        return -1;
    Model m;
    m.nctrs = ncounters;
    m.ctr_expected = counter_reductions;
    m.nbars = nbars;
    m.nbufs = nbufs;
    m.nroles = nroles;
    m.expected = bar_expected;
    m.group = role_group;
    m.off = role_offsets;
    m.ops = ops;
    std::vector<std::string> nm = split_lines(names);
    if (static_cast<int>(nm.size()) < nroles + nbars + nbufs) nm.resize(nroles + nbars + nbufs, "?");
    m.role_name.assign(nm.begin(), nm.begin() + nroles);
    m.bar_name.assign(nm.begin() + nroles, nm.begin() + nroles + nbars);
    m.buf_name.assign(nm.begin() + nroles + nbars, nm.begin() + nroles + nbars + nbufs);
    m.o_pc = 0;
    m.o_bar = nroles;
    m.o_buf = m.o_bar + 3 * nbars;
    m.o_mq = m.o_buf + nbufs;
    m.o_asy = m.o_mq + 1 + kMaxQueue;
    m.o_ctr = m.o_asy + 1 + kMaxAsync;
    m.len = m.o_ctr + 2 * ncounters;
    Checker c(m, max_states);
    const int rc = c.run();
    if (states_out) *states_out = c.states;
    snprintf(msg, static_cast<size_t>(msg_len), "%s", c.msg.c_str());
    return rc;
}

extern "C" int32_t ts_protocol_check(int32_t nbars, const int32_t *bar_expected, int32_t nbufs, int32_t nroles,
                                     const int32_t *role_group, const int32_t *role_offsets, const int32_t *ops,
                                     const char *names, int64_t max_states, int64_t *states_out, char *msg,
                                     int32_t msg_len) {
    return ts_protocol_check_ex(nbars, bar_expected, nbufs, nroles, role_group, role_offsets, ops, 0, nullptr, names,
                                max_states, states_out, msg, msg_len);
}
