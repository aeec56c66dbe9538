"""Index arithmetic of the kernels, checked on the CPU (no GPU needed).

compute-sanitizer is not available here, so the address formulas of the
kernels whose indexing is least obvious are restated in Python and checked
exhaustively over shape classes:

* the row-class kernel: every raw TMA box lands inside its raw stage,
  128-byte aligned and disjoint from the others; every read of the realign
  step stays inside the box it belongs to; every 16-byte chunk of the
  swizzled stage is written exactly once per K block;
* the row-class maps: each class map starts at the 16-byte boundary at or
  below its first row (so inside the matrix's allocation), its rows all sit
  the same delta < 8 elements past that boundary, its pitch is a multiple of
  16 bytes, and it ends at the last row's end;
* the even split of a send list over CTAs used by the exchange kernels;
* the fused kernels' tile raster: one to one onto the launch's output tiles;
* the repack kernel: every 32-bit word it loads holds a byte of the row being
  copied (so it lies inside the row's 16-byte granules, inside the
  allocation), every word it stores lies inside the destination row's pitch,
  and the copied elements come out exactly, with a zero padding element for
  odd lengths.

The constants and formulas mirror fused_tcr.cu, ia2av.cu and repack.cu; a
change there must be made here too.
"""
import itertools

import numpy as np
import pytest

KROW, NROW, BK, BM_CTA, BN_CTA = 144, 272, 64, 128, 128
RAW_A = BM_CTA * KROW
RAW_B = BN_CTA * KROW
SW_A, SW_B, B_BOX = 16384, 16384, 8192


def _classes(rowlen, aligned=True, pitch=None, base_off=None):
    """Row classes as fused_tcr.cu's row_classes counts them: n rows span a
    multiple of 16 bytes and n * pitch covers the row plus the largest delta."""
    pitch = rowlen if pitch is None else pitch
    base_off = (0 if aligned else 2) if base_off is None else base_off
    n = 1
    while (pitch * 2 * n) % 16:
        n *= 2
    while n < 8 and n * pitch < rowlen + max(((base_off + q * pitch * 2) % 16) // 2
                                             for q in range(n)):
        n *= 2
    return n


def _stage_addresses(wt, ncx, ncw):
    """(raw boxes, realign reads and writes) of one CTA and K block."""
    lgx, lgw = ncx.bit_length() - 1, ncw.bit_length() - 1
    boxes = [(b * (RAW_A >> lgx), (BM_CTA // ncx) * KROW) for b in range(ncx)]
    if wt:
        boxes += [(RAW_A + b * (RAW_B >> lgw), (BN_CTA // ncw) * KROW) for b in range(ncw)]
    else:
        boxes += [(RAW_A + b * ((BK * NROW) >> lgw), (BK // ncw) * NROW) for b in range(ncw)]
    sx, sw = 5 - lgx, 5 - lgw
    steps = []
    for bt in range(16):                       # 16 batches of four warp steps
        for s in range(4):
            for lane in range(32):
                rg, c = lane >> 3, lane & 7
                if bt < 8:
                    it0 = bt * 4
                    b, v0 = it0 >> sx, it0 & ((1 << sx) - 1)
                    j = 4 * (v0 + s) + rg
                    i = b + (j << lgx)
                    box = b * (RAW_A >> lgx)
                    src, box_end = box + j * KROW + c * 16, box + (BM_CTA // ncx) * KROW
                    dst = i * 128 + ((c ^ (i & 7)) << 4)
                elif wt:
                    it0 = (bt - 8) * 4
                    b, v0 = it0 >> sw, it0 & ((1 << sw) - 1)
                    j = 4 * (v0 + s) + rg
                    i = b + (j << lgw)
                    box = RAW_A + b * (RAW_B >> lgw)
                    src, box_end = box + j * KROW + c * 16, box + (BN_CTA // ncw) * KROW
                    dst = SW_A + i * 128 + ((c ^ (i & 7)) << 4)
                else:
                    it0 = (bt - 8) * 4
                    b, v0 = it0 >> sw, it0 & ((1 << sw) - 1)
                    j = 2 * (v0 + s) + (rg >> 1)
                    half, kr = rg & 1, b + (j << lgw)
                    box = RAW_A + b * ((BK * NROW) >> lgw)
                    src = box + j * NROW + (half * 8 + c) * 16
                    box_end = box + (BK // ncw) * NROW
                    dst = SW_A + half * B_BOX + kr * 128 + ((c ^ (kr & 7)) << 4)
                steps.append((src, box_end, dst))
    return boxes, steps


@pytest.mark.parametrize("wt", [0, 1])
@pytest.mark.parametrize("ncx,ncw", list(itertools.product((1, 2, 4, 8), repeat=2)))
def test_row_class_stage_addressing(wt, ncx, ncw):
    boxes, steps = _stage_addresses(wt, ncx, ncw)
    for off, size in boxes:
        assert off % 128 == 0 and off + size <= RAW_A + RAW_B
    for (o1, s1), (o2, _) in zip(sorted(boxes), sorted(boxes)[1:]):
        assert o1 + s1 <= o2
    written = {}
    for src, box_end, dst in steps:
        assert src % 16 == 0 and src + 32 <= box_end       # both granules of the shift
        assert dst % 16 == 0 and dst + 16 <= SW_A + SW_B
        written[dst] = written.get(dst, 0) + 1
    assert len(written) == (SW_A + SW_B) // 16 and set(written.values()) == {1}


def _tile_coord(tile, m_tiles, n_tiles, group_m):
    """tc_ptx.cuh's tile_coord: group, then super-rows of group_m m tiles
    walked n tile by n tile (group_m <= 0: row-major)."""
    per_group = m_tiles * n_tiles
    g, t = divmod(tile, per_group)
    if group_m <= 0:
        return g, t // n_tiles, t % n_tiles
    span = group_m * n_tiles
    sr, u = divmod(t, span)
    first_m = sr * group_m
    rows = min(group_m, m_tiles - first_m)
    return g, first_m + u % rows, u // rows


@pytest.mark.parametrize("group_m", [0, 1, 4, 8, 16])
def test_tile_raster_covers_every_tile_once(group_m):
    """The persistent fused kernels hand tile t to pair t mod npairs and place
    it with tile_coord: over any shape (ragged last super-row included) the
    tiles of a launch map one to one onto (group, m tile, n tile), so every
    output tile is computed exactly once."""
    for m_tiles in range(1, 37):
        for n_tiles in range(1, 19):
            groups = 3
            seen = set()
            for tile in range(groups * m_tiles * n_tiles):
                g, mt, nt = _tile_coord(tile, m_tiles, n_tiles, group_m)
                assert 0 <= g < groups and 0 <= mt < m_tiles and 0 <= nt < n_tiles
                seen.add((g, mt, nt))
            assert len(seen) == groups * m_tiles * n_tiles


def _class_map(base, rowlen, nrows, n, q, rpitch=None):
    """(map base address, delta, inner extent, outer extent, pitch) of class q
    of a matrix whose rows are `rpitch` elements apart (default: dense)."""
    rpitch = rowlen if rpitch is None else rpitch
    a = base + q * rpitch * 2
    a16 = a & ~15
    d = (a - a16) // 2
    return a16, d, rowlen + d, (nrows - q + n - 1) // n, rpitch * 2 * n


@pytest.mark.parametrize("rowlen", [1, 2, 3, 4, 5, 6, 7, 8, 9, 65, 100, 257, 1025, 2050, 4100,
                                    65535])
@pytest.mark.parametrize("base_off", [0, 2, 4, 6, 8, 10, 12, 14])
@pytest.mark.parametrize("extra", [0, 1, 3, 8])            # caller pitch = rowlen + extra
def test_row_class_maps_stay_inside_the_matrix(rowlen, base_off, extra):
    base = (1 << 20) + base_off                           # an element-aligned pointer
    alloc_start = base & ~15                              # allocations start 16-byte aligned
    nrows = 37
    rpitch = rowlen + extra
    end = base + ((nrows - 1) * rpitch + rowlen) * 2      # the pitched matrix's last byte + 1
    n = _classes(rowlen, pitch=rpitch, base_off=base_off)
    for q in range(min(n, nrows)):
        a16, d, inner, outer, pitch = _class_map(base, rowlen, nrows, n, q, rpitch)
        assert a16 >= alloc_start and 0 <= d < 8 and pitch % 16 == 0
        assert pitch >= inner * 2                          # rows do not overlap in the map
        for j in range(outer):
            row = q + j * n
            start = base + row * rpitch * 2
            assert start - (a16 + j * pitch) == 2 * d      # every row sits delta past its boundary
        last = q + (outer - 1) * n
        assert a16 + (outer - 1) * pitch + inner * 2 == base + (last * rpitch + rowlen) * 2 <= end


@pytest.mark.parametrize("n", [0, 1, 5, 17, 1000, 2 ** 40 + 7])
@pytest.mark.parametrize("parts", [1, 3, 38, 152, 1216])
def test_even_split_covers_the_send_list(n, parts):
    q, rem = divmod(n, parts)
    prev = 0
    for part in range(parts):
        lo = q * part + min(part, rem)
        hi = lo + q + (1 if part < rem else 0)
        assert lo == prev and hi >= lo
        prev = hi
    assert prev == n


def _repack_row(mem, sa, length, pitch, unroll=16):
    """One warp's copy of one row, as repack.cu computes it (byte addresses
    into `mem`, a bytes-like view of memory starting at address 0): returns
    the destination words and the set of source word indices loaded."""
    wa = sa & ~3
    odd = (sa & 3) != 0
    end = sa + 2 * length
    nsrc = (end - wa + 3) >> 2
    nout = (length + 1) >> 1
    word = lambda k: int.from_bytes(mem[wa + 4 * k: wa + 4 * k + 4], "little")
    loaded, out = set(), {}
    for base in range(0, nout, 32 * unroll):
        for u in range(unroll):
            v, nb = [], []
            for lane in range(32):
                k = base + u * 32 + lane
                if k < nsrc:
                    loaded.add(k)
                v.append(word(k) if k < nsrc else 0)
            if odd:
                for lane in range(32):
                    k1 = base + u * 32 + lane + 1
                    if lane < 31:
                        nb.append(v[lane + 1])
                    else:
                        if k1 < nsrc:
                            loaded.add(k1)
                        nb.append(word(k1) if k1 < nsrc else 0)
                v = [((a >> 16) | (b << 16)) & 0xFFFFFFFF for a, b in zip(v, nb)]
            for lane in range(32):
                k = base + u * 32 + lane
                if k < nout:
                    w = v[lane]
                    if (length & 1) and k == nout - 1:
                        w &= 0xFFFF
                    out[k] = w
    return out, loaded, nsrc, wa


@pytest.mark.parametrize("length", [1, 2, 3, 7, 8, 9, 63, 64, 65, 255, 256, 257, 300])
@pytest.mark.parametrize("off", [0, 2, 4, 6, 8, 10, 12, 14])
def test_repack_reads_inside_the_row_and_copies_exactly(length, off):
    rng = np.random.default_rng(length * 16 + off)
    nrows = 3
    base = 4096 + off                                     # element-aligned matrix start
    mem = bytearray(rng.integers(0, 256, size=base + nrows * length * 2 + 64, dtype=np.uint8))
    elems = np.frombuffer(bytes(mem[base:base + nrows * length * 2]), dtype="<u2").reshape(
        nrows, length)
    pitch = (length + 63) // 64 * 64
    for row in range(nrows):
        sa = base + row * length * 2
        out, loaded, nsrc, wa = _repack_row(mem, sa, length, pitch)
        for k in loaded:                                  # each loaded word holds a row byte
            assert wa + 4 * k < sa + 2 * length and wa + 4 * k + 4 > sa
        assert max(out) < pitch // 2 + (pitch % 2)        # stores stay inside the pitch
        got = np.array([out[k] for k in sorted(out)], dtype=np.uint32)
        halves = np.stack([got & 0xFFFF, got >> 16], axis=1).reshape(-1)
        np.testing.assert_array_equal(halves[:length], elems[row])
        if length & 1:
            assert halves[length] == 0


def _element_epilogue_stores(delta):
    """(offset, size) of every global store the element-wise epilogue makes
    for one run, in bytes from the run's 16-byte aligned start, as
    tcu_epilogue.cuh computes them: chunks 1..7 whole, chunk 0 whole or its
    head [2 delta, 16), chunk 8's tail [0, 2 delta) at offset 128."""
    lo = 2 * delta
    stores = [(16 * k, 16) for k in range(1, 8)]
    if lo == 0:
        stores.append((0, 16))
        return stores
    b = lo
    if b & 2:
        stores.append((b, 2))
        b += 2
    if b & 4:
        stores.append((b, 4))
        b += 4
    if b & 8:
        stores.append((b, 8))
    if lo & 8:
        stores.append((128, 8))
    if lo & 4:
        stores.append((128 + (lo & 8), 4))
    if lo & 2:
        stores.append((128 + (lo & 12), 2))
    return stores


@pytest.mark.parametrize("delta", range(8))
def test_element_epilogue_writes_each_run_byte_once(delta):
    lo = 2 * delta
    written = np.zeros(160, dtype=np.int64)
    for off, size in _element_epilogue_stores(delta):
        assert off % size == 0                       # every store aligned to its size
        assert off + size <= 144                     # inside the staged row buffer
        written[off:off + size] += 1
    want = np.zeros(160, dtype=np.int64)
    want[lo:lo + 128] = 1                            # the run, and nothing else
    np.testing.assert_array_equal(written, want)


@pytest.mark.parametrize("delta", range(8))
def test_element_epilogue_staging_shift(delta):
    """Staged word q + i = funnel-shift of (w[i-1], w[i]) by 16 (odd delta)
    or 32 (even): buffer element k holds column k - delta."""
    w = [(2 * i) | ((2 * i + 1) << 16) for i in range(32)]      # columns 0..63, packed
    sh = 16 if delta & 1 else 32
    fsr = lambda lo_, hi_, s: (((hi_ << 32) | lo_) >> min(s, 32)) & 0xFFFFFFFF
    q = delta >> 1
    buf = [None] * 36
    buf[q] = fsr(0, w[0], sh)
    for i in range(1, 32):
        buf[q + i] = fsr(w[i - 1], w[i], sh)
    buf[q + 32] = fsr(w[31], 0, sh)
    elems = []
    for wd in buf:
        elems += [None, None] if wd is None else [wd & 0xFFFF, wd >> 16]
    assert elems[delta:delta + 64] == list(range(64))


# ---------------------------------------------------------------------------
# all_to_all_v kernel (a2av.cu): block ranges, segments, staged chunks, the
# warps' chunk shares and the piece writes.
A2AV_CHUNKS, A2AV_PAD, A2AV_WARPS, A2AV_MAXSEG = (6144, 4096), 128, 16, 4
P_MAX = 64   # pieces tabled per segment (the kernel's kA2avMaxP)


def _a2av_block_copy(sc, es, in_base, in_len_b, out_base, nb, chunk, mem, out_mem, written):
    """Run the kernel's addressing for every block: `mem` maps a source
    address to its byte value, `out_mem` / `written` receive the stores.
    Checks every staged read, every direct read and every store against the
    buffers."""
    P = sc.shape[0]
    rowtot = sc.sum(axis=1)
    T = int(rowtot.sum())
    rowoff = np.concatenate([[0], np.cumsum(rowtot)[:-1]])
    sd = np.concatenate([np.zeros((P, 1), np.int64), np.cumsum(sc, axis=1)[:, :-1]], axis=1)
    rd = np.concatenate([np.zeros((1, P), np.int64), np.cumsum(sc, axis=0)[:-1, :]], axis=0)
    span = [(in_base[r], in_base[r] + int(in_len_b[r])) for r in range(P)]
    for b in range(nb):
        q_, rem = divmod(T, nb)
        lo, hi = q_ * b + min(b, rem), q_ * (b + 1) + min(b + 1, rem)
        segs = []
        for r in range(P):
            off, tot = int(rowoff[r]), int(rowtot[r])
            if tot > 0 and off < hi and off + tot > lo:
                slo, shi = max(lo - off, 0), min(hi - off, tot)
                g0 = (in_base[r] + slo * es) & ~15
                g1 = (in_base[r] + shi * es + 15) & ~15
                segs.append((r, slo, shi, g0, g1, -(-(g1 - g0) // chunk)))
        chbase = np.concatenate([[0], np.cumsum([s[5] for s in segs])]).astype(np.int64)
        # Loads: chunk t of the block staged from [c0, ce).
        staged = {}
        t = 0
        for (r, slo, shi, g0, g1, nch) in segs:
            lo_g, hi_g = in_base[r] & ~15, (in_base[r] + in_len_b[r] + 15) & ~15
            for c0 in range(g0, g1, chunk):
                ce = min(c0 + chunk + 16, g1)
                assert lo_g <= c0 < ce <= hi_g and (ce - c0) % 16 == 0 and c0 % 16 == 0
                assert ce - c0 <= (chunk + A2AV_PAD)
                staged[t] = (c0, ce)
                t += 1
        assert t == chbase[-1]
        # Batch by batch: tables (head and tail bytes copied from the send
        # buffer), then each warp's chunks t = w, w + A2AV_WARPS, ...
        for b0 in range(0, len(segs), A2AV_MAXSEG):
            batch = segs[b0:b0 + A2AV_MAXSEG]
            tables = []
            pieces = {}
            for (i, slo, shi, g0, g1, nch) in batch:
                runs = []
                for j in range(P):
                    c = int(sc[i, j])
                    c0e, c1e = max(slo, sd[i, j]), min(shi, sd[i, j] + c)
                    n = (c1e - c0e) * es if c1e > c0e else 0
                    if n == 0:
                        continue
                    src = in_base[i] + c0e * es
                    dst = out_base[j] + (rd[i, j] + (c0e - sd[i, j])) * es
                    head = min((16 - dst % 16) % 16, n)
                    nvec, tail = (n - head) >> 4, (n - head) & 15
                    pieces[(len(tables), j)] = (src + head, dst + head, nvec, head, tail)
                    if nvec > 0:
                        runs.append((src + head, dst + head, nvec))
                tables.append(runs)
            # Head and tail bytes: byte slot x = (piece, b) of the batch, b < 15
            # the head's byte b, 16 <= b < 31 the tail's byte b - 16.
            for x in range(len(batch) * P_MAX * 32):
                key = ((x >> 5) // P_MAX, (x >> 5) % P_MAX)
                if key not in pieces:
                    continue
                vb, d, nvec, head, tail = pieces[key]
                bb = x & 31
                if bb < head:
                    o = bb - head
                elif 16 <= bb < 16 + tail:
                    o = nvec * 16 + bb - 16
                else:
                    continue
                assert span[segs[b0 + key[0]][0]][0] <= vb + o < span[segs[b0 + key[0]][0]][1]
                out_mem[d + o] = mem[vb + o]
                written[d + o] += 1
            tb, te = chbase[b0], chbase[b0 + len(batch)]
            for g in range(A2AV_WARPS):
                t = tb + ((g - tb % A2AV_WARPS) + A2AV_WARPS) % A2AV_WARPS
                sg, q = b0, 0
                while t < te:
                    while chbase[sg + 1] <= t:
                        sg, q = sg + 1, 0
                    c0s, ce = staged[t]
                    G1 = segs[sg][4]
                    c0 = segs[sg][3] + (t - chbase[sg]) * chunk
                    assert c0 == c0s
                    c1 = min(c0 + chunk, G1)
                    stage = mem[c0:ce]
                    runs = tables[sg - b0]
                    qq = q
                    while qq < len(runs):
                        vb, d, nvec = runs[qq]
                        if vb >= c1:
                            break
                        last = vb + (nvec - 1) * 16
                        if last < c0:
                            q = qq + 1
                            qq += 1
                            continue
                        vlo = 0 if vb >= c0 else (c0 - vb + 15) >> 4
                        vhi = min((c1 - vb + 15) >> 4, nvec)
                        o = vb + vlo * 16 - c0
                        k = np.arange(vhi - vlo)
                        rd0 = (o & ~15) + 16 * k          # first staged word read
                        assert rd0.min() >= 0 and (rd0 + 32).max() <= (chunk + A2AV_PAD)
                        first = o + 16 * k                # the vector's bytes in the stage
                        assert (first + 16).max() <= ce - c0
                        dv = d + 16 * (vlo + k)
                        assert (dv % 16 == 0).all()
                        idx = (first[:, None] + np.arange(16)).ravel()
                        dd = (dv[:, None] + np.arange(16)).ravel()
                        out_mem[dd] = stage[idx]
                        written[dd] += 1
                        if last >= c1:
                            break
                        q = qq + 1
                        qq += 1
                    t += A2AV_WARPS


@pytest.mark.parametrize("chunk", A2AV_CHUNKS)
@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("es", [1, 4])
def test_exchange_block_addressing(seed, es, chunk):
    """Every byte each rank receives is written exactly once with the right
    source byte, staged reads stay inside the staged chunk (and its ring
    slot), bulk loads stay inside the send buffer's 16-byte granules, and no
    byte outside the received ranges is stored -- for launch widths below,
    at and above P, unaligned bases and pieces spanning chunks."""
    rng = np.random.default_rng(seed)
    P = int(rng.choice([1, 2, 3, 5, 8]))
    small = rng.integers(0, 40, size=(P, P))
    big = rng.integers(0, 12 * chunk // es, size=(P, P))
    sc = np.where(rng.random((P, P)) < 0.4, big, small).astype(np.int64)
    sc[rng.random((P, P)) < 0.2] = 0
    in_len = sc.sum(axis=1) * es
    out_len = sc.sum(axis=0) * es
    # Buffers at 4096-byte-spaced slots plus an offset of whole elements.
    addr = 4096
    in_base, out_base = [], []
    for n in in_len:
        addr += int(rng.integers(0, 16 // es)) * es
        in_base.append(addr)
        addr = (addr + int(n) + 4096 + 4095) // 4096 * 4096
    for n in out_len:
        addr += int(rng.integers(0, 16 // es)) * es
        out_base.append(addr)
        addr = (addr + int(n) + 4096 + 4095) // 4096 * 4096
    mem = rng.integers(0, 256, size=addr + 64).astype(np.uint8)
    out_mem = np.zeros(addr + 64, np.uint8)
    written = np.zeros(addr + 64, np.int32)
    for nb in sorted({1, 3, max(1, P - 1), P, 2 * P + 1, 64}):
        out_mem[:] = 0
        written[:] = 0
        _a2av_block_copy(sc, es, in_base, in_len, out_base, nb, chunk, mem, out_mem, written)
        expect_w = np.zeros_like(written)
        for j in range(P):
            expect_w[out_base[j]:out_base[j] + out_len[j]] = 1
        assert np.array_equal(written, expect_w), nb
        for i in range(P):
            for j in range(P):
                sdb = int(sc[i, :j].sum()) * es
                rdb = int(sc[:i, j].sum()) * es
                n = int(sc[i, j]) * es
                assert np.array_equal(out_mem[out_base[j] + rdb:out_base[j] + rdb + n],
                                      mem[in_base[i] + sdb:in_base[i] + sdb + n]), (nb, i, j)


def _ring_schedule(stages, groups, nchunks, rng):
    """One random interleaving of the exchange's ring protocol: producer g
    loading chunks t = g, g + groups, ... in order into stage t % stages
    after a parity wait on the stage's empty barrier, loads landing at
    random later times (completing a phase of the stage's full barrier),
    and consumer group t % groups taking chunk t after a parity wait on the
    full barrier, then arriving on the empty barrier.  A parity wait on
    phase u passes when the number of completed phases has the other parity
    (mbarrier try_wait.parity).  Returns False when a group passed its wait
    while its stage held another chunk or had a load in flight, or a
    producer loaded into a stage with a load still in flight."""
    full_c = [0] * stages
    empty_c = [0] * stages
    content = [-1] * stages
    in_flight = {}                       # stage -> chunk
    issue = [list(range(g, nchunks, groups)) for g in range(groups)]
    todo = [list(range(g, nchunks, groups)) for g in range(groups)]
    while any(issue) or in_flight or any(todo):
        moves = []
        for g in range(groups):
            if issue[g]:
                t = issue[g][0]
                s, u = t % stages, t // stages
                if (empty_c[s] & 1) != ((u & 1) ^ 1):
                    moves.append(("issue", g))
        moves += [("land", s) for s in in_flight]
        for g in range(groups):
            if todo[g]:
                t = todo[g][0]
                s, u = t % stages, t // stages
                if (full_c[s] & 1) != (u & 1):
                    moves.append(("take", g))
        if not moves:
            return False                 # nobody can move: a deadlock
        kind, arg = moves[rng.integers(len(moves))]
        if kind == "issue":
            t = issue[arg].pop(0)
            s = t % stages
            if s in in_flight:
                return False
            in_flight[s] = t
        elif kind == "land":
            content[arg] = in_flight.pop(arg)
            full_c[arg] += 1
        else:
            t = todo[arg].pop(0)
            s = t % stages
            if content[s] != t or s in in_flight:
                return False
            empty_c[s] += 1
    return True


def test_exchange_ring_protocol_under_random_schedules():
    """The kernel's slots: warp w's i-th chunk goes to its slot i % S, so
    chunk t sits in slot t % (W * S) of the block when slots are numbered
    warp-major.  With the slot count a multiple of the pipelines (W * S),
    every slot has one loader and one consumer, and no pipeline ever reads a
    slot before its own chunk has landed there, under any interleaving; with
    other slot counts some interleaving breaks the protocol."""
    rng = np.random.default_rng(0)
    for stages in (A2AV_WARPS * 2, A2AV_WARPS * 3):
        for _ in range(100):
            assert _ring_schedule(stages, A2AV_WARPS, int(rng.integers(1, 200)), rng)
    for stages in (6, 12):
        for _ in range(100):
            assert _ring_schedule(stages, 3, int(rng.integers(1, 60)), rng)
    for stages in (A2AV_WARPS * 2 + 1, 11):
        assert not all(_ring_schedule(stages, 4 if stages == 11 else A2AV_WARPS, 200, rng)
                       for _ in range(100))


@pytest.mark.parametrize("pairs_per_cluster", [1, 2])
@pytest.mark.parametrize("group_m", [0, 4, 16])
def test_cluster_super_tiles_cover_every_tile_once(pairs_per_cluster, group_m):
    """fused_tc2.cu with CL pairs per cluster: super-tile st (CL m tiles of one
    n tile, walked by tile_coord with super-rows of group_m / CL) gives pair
    pc the m tile CL * mt' + pc.  Every output tile is computed by exactly
    one (super-tile, pair); the only extra work is the second pair's tile
    past the last m tile when the m-tile count is odd, which the kernel
    loads as zeros and does not store."""
    CL = pairs_per_cluster
    gs = group_m // CL if group_m // CL > 0 else 1   # kGroupS of the kernel
    for m_tiles in range(1, 21):
        for n_tiles in range(1, 9):
            groups = 2
            m_super = (m_tiles + CL - 1) // CL
            seen, extra = {}, 0
            for st in range(groups * m_super * n_tiles):
                g, ms, nt = _tile_coord(st, m_super, n_tiles, gs)
                for pc in range(CL):
                    mt = ms * CL + pc
                    if mt >= m_tiles:
                        extra += 1
                        continue
                    seen[(g, mt, nt)] = seen.get((g, mt, nt), 0) + 1
            assert len(seen) == groups * m_tiles * n_tiles and set(seen.values()) == {1}
            assert extra == (groups * n_tiles if CL == 2 and m_tiles % 2 else 0)
