"""Brute-force restatement of the dispatch layout, used to pin the oracle.

Placement is defined here by sorting every (source rank s, token t, slot k) pair with
an explicit key and counting with explicit predicates, not by running counters and
prefix scans as the oracle does:

* send order on rank s:          key (expert, t, k)
* receive order on rank d:       key (s, expert, t, k) over pairs whose expert d hosts
* grouped order of expert e:     key (s, t, k)
* every offset is a count of the pairs that sort before, by its own predicate.

Pure Python loops, for tiny shapes only.
"""
from __future__ import annotations

import numpy as np


def layout(N, T, E, R, cap, idx):
    L = E // N
    cap = cap if cap > 0 else N * T
    RB = N * T * max(R, L)
    idx = np.asarray(idx).reshape(N, T, R)
    pairs = []          # (s, t, k, e) with a valid expert
    status = 0
    for s in range(N):
        for t in range(T):
            for k in range(R):
                e = int(idx[s, t, k])
                if 0 <= e < E:
                    pairs.append((s, t, k, e))
                else:
                    status |= 1 << 2
    owner = lambda e: e // L
    cnt = np.zeros((N, E), np.int32)
    soff = np.zeros((N, E), np.int32)
    for s in range(N):
        for e in range(E):
            cnt[s, e] = sum(1 for p in pairs if p[0] == s and p[3] == e)
            soff[s, e] = sum(1 for p in pairs if p[0] == s and p[3] < e)
    C = np.zeros((N, N), np.int32)
    roff = np.zeros((N, N), np.int32)
    rtot = np.zeros((N,), np.int32)
    for d in range(N):
        rtot[d] = sum(1 for p in pairs if owner(p[3]) == d)
        for s in range(N):
            C[s, d] = sum(1 for p in pairs if p[0] == s and owner(p[3]) == d)
            roff[d, s] = sum(1 for p in pairs if p[0] < s and owner(p[3]) == d)
    ecnt = np.zeros((N, L), np.int32)
    eoff = np.zeros((N, L, N), np.int32)
    for d in range(N):
        for l in range(L):
            e = d * L + l
            ecnt[d, l] = sum(1 for p in pairs if p[3] == e)
            if ecnt[d, l] > cap:
                status |= 1 << 3
            for s in range(N):
                eoff[d, l, s] = sum(1 for p in pairs if p[3] == e and p[0] < s)
    pos = np.full((N, T, R), -1, np.int32)
    rrow = np.full((N, T, R), -1, np.int32)
    slot = np.full((N, T, R), -1, np.int32)
    slot_src = np.full((N, L, cap), -1, np.int32)
    recv_src = np.full((N, RB), -1, np.int32)
    pid = lambda p: (p[0] * T + p[1]) * R + p[2]
    for s in range(N):
        mine = sorted((p for p in pairs if p[0] == s), key=lambda p: (p[3], p[1], p[2]))
        for i, p in enumerate(mine):
            pos[p[0], p[1], p[2]] = i
    for d in range(N):
        mine = sorted((p for p in pairs if owner(p[3]) == d), key=lambda p: (p[0], p[3], p[1], p[2]))
        for i, p in enumerate(mine):
            rrow[p[0], p[1], p[2]] = i
            recv_src[d, i] = pid(p)
    for e in range(E):
        d, l = e // L, e % L
        mine = sorted((p for p in pairs if p[3] == e), key=lambda p: (p[0], p[1], p[2]))
        for i, p in enumerate(mine):
            if i < cap:
                slot[p[0], p[1], p[2]] = i
                slot_src[d, l, i] = pid(p)
    return dict(cnt=cnt, C=C, soff=soff, roff=roff, rtot=rtot, ecnt=ecnt, eoff=eoff, pos=pos,
                rrow=rrow, slot=slot, slot_src=slot_src, recv_src=recv_src, status=status)


LAYOUT_KEYS = ("cnt", "C", "soff", "roff", "rtot", "ecnt", "eoff", "pos", "rrow", "slot",
               "slot_src", "recv_src")
