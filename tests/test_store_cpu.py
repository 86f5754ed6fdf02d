"""The storage tier on the host (no GPU): expert files and the host tier.

* moe_store_write lays a layer's routed experts out as the header says: a
  4096-byte header, then expert e at 4096 + e * stride, stride = the blob size
  rounded up to 4096, zero padded; each expert's region holds that expert's
  scale/bias words at the places the blob layout puts them and exactly that
  expert's 4-bit codes (as a multiset: the blob permutes nibbles in a word);
* moe_store_fetch returns the file's bytes (read here independently with
  numpy), with or without O_DIRECT;
* the tier reuses the unpinned entry whose expert was fetched least often
  (ties: least recently used), never a pinned one (MOE_EBUSY when all are
  pinned); readahead fills free entries, never evicts an expert read ahead
  and not yet used, and displaces only experts fetched no more often;
* failures: wrong shapes, foreign or short files, a read past a file that
  shrank after opening (MOE_EIO; a later fetch retries), a read cut short
  inside an expert (the entry fails whole, also when read in pieces);
* reads split into pieces over several readers give the same bytes;
* several host threads fetching at once get the right bytes.
"""
import os
import threading

import numpy as np
import pytest

import expert_streaming_ffn_gb300 as moe
import synth

# d=512, 8 experts, I=192: the blob (165,888 B) is not a multiple of 4096, so
# every expert carries padding
SHAPES = synth.Shapes(512, 8, 2, 192, 512, synth.GELU_TANH)
ALIGN = 4096


@pytest.fixture(scope="module")
def weights():
    return synth.layer_weights(SHAPES, 3, 5)


@pytest.fixture()
def expert_file(tmp_path, weights):
    p = str(tmp_path / "layer3.experts")
    moe.moe_store_write(p, SHAPES, weights)
    return p


def _region(path, e):
    stride = moe.moe_store_expert_stride(SHAPES)
    raw = np.fromfile(path, np.uint8)
    return raw[ALIGN + e * stride: ALIGN + (e + 1) * stride]


def _nibbles(codes):
    c = np.asarray(codes, np.uint8).reshape(-1)
    return np.bincount(np.concatenate([c & 15, c >> 4]), minlength=16)


def _words(scale, bias):
    return np.asarray(scale, np.uint32) | (np.asarray(bias, np.uint32) << 16)


# position of row r's scale word within a 32-word block: 4 (r % 8) + r // 8
SB_ROW = np.array([4 * (r % 8) + r // 8 for r in range(32)])


def test_file_layout_header_and_padding(expert_file):
    eb = moe.moe_expert_bytes(SHAPES)
    stride = moe.moe_store_expert_stride(SHAPES)
    assert eb == synth.expert_bytes(SHAPES) == 165888
    assert stride == 41 * ALIGN and stride % ALIGN == 0 and stride >= eb
    raw = np.fromfile(expert_file, np.uint8)
    assert raw.size == ALIGN + SHAPES.n_experts * stride
    assert bytes(raw[:8]) == b"MOEXPRTS"
    hdr = raw[:ALIGN]
    assert int(hdr[8:12].view(np.uint32)[0]) == 1 and int(hdr[12:16].view(np.uint32)[0]) == ALIGN
    shp = hdr[16:40].view(np.int32)
    assert list(shp) == [SHAPES.d_model, SHAPES.n_experts, SHAPES.top_k, SHAPES.d_ff, SHAPES.d_ff_shared,
                         SHAPES.act]
    assert list(hdr[48:72].view(np.uint64)) == [eb, stride, ALIGN]
    for e in range(SHAPES.n_experts):
        assert not _region(expert_file, e)[eb:].any(), "padding must be zero"


def test_each_region_holds_its_expert(expert_file, weights):
    d, I = SHAPES.d_model, SHAPES.d_ff
    gu = I * d // 2 + I * d // 16  # one gate or up matrix
    for e in range(SHAPES.n_experts):
        r = _region(expert_file, e)
        (gc, gs, gb), (uc, us, ub), (dc, ds, db) = weights.expert(e)
        for m, (c, s, b) in enumerate([(gc, gs, gb), (uc, us, ub)]):
            # records of 1152 bytes per (32-row tile, group of 64): 32 lanes x
            # 2 chunks x 16 code bytes, then one scale|bias word per lane
            rec = r[m * gu:(m + 1) * gu].reshape(I // 32, d // 64, 1152)
            words = rec[:, :, 1024:].copy().view(np.uint32)[:, :, SB_ROW]  # [rt][g][row]
            want = _words(s, b).reshape(I // 32, 32, d // 64).transpose(0, 2, 1)
            assert (words == want).all(), (e, m)
            assert (_nibbles(rec[:, :, :1024]) == _nibbles(c)).all(), (e, m)
        # down, column-sliced: all codes first, then the words as 128-byte
        # blocks ordered by (group, row tile)
        dn = r[2 * gu:2 * gu + d * I // 2 + d * I // 16]
        words = dn[d * I // 2:].copy().view(np.uint32).reshape(I // 64, d // 32, 32)[:, :, SB_ROW]
        want = _words(ds, db).reshape(d // 32, 32, I // 64).transpose(2, 0, 1)
        assert (words == want).all(), e
        assert (_nibbles(dn[:d * I // 2]) == _nibbles(dc)).all(), e


@pytest.mark.parametrize("chunk", [0, 4096, 65536])
@pytest.mark.parametrize("flags", [0, moe.MOE_STORE_DIRECT])
def test_fetch_returns_the_files_bytes(expert_file, flags, chunk):
    # whole-expert reads, and reads in pieces of 4 KiB (41 of them) and 64 KiB
    # (two full pieces and a 36 KiB tail) spread over the readers
    eb = moe.moe_expert_bytes(SHAPES)
    st = moe.moe_store_open(expert_file, SHAPES, 3, 2, flags)
    moe.moe_store_set_read_chunk(st, chunk)
    try:
        for e in [5, 0, 7, 5, 2]:
            got = moe.moe_store_fetch(st, e, eb)
            assert (got == _region(expert_file, e)[:eb]).all(), e
            moe.moe_store_release(st, e)
        s = moe.moe_store_get_stats(st)
        assert s["fetches"] == 5 and s["tier_hits"] == 1 and s["reads"] == 4
        assert s["bytes_read"] == 4 * moe.moe_store_expert_stride(SHAPES)
        assert s["direct"] in (0, 1) and (flags or s["direct"] == 0)
    finally:
        moe.moe_store_close(st)


def test_tier_evicts_the_least_fetched_then_least_recent_entry(expert_file):
    eb = moe.moe_expert_bytes(SHAPES)
    st = moe.moe_store_open(expert_file, SHAPES, 2, 1)
    try:
        def use(e):
            moe.moe_store_fetch(st, e, eb)
            moe.moe_store_release(st, e)

        def tier():
            return sorted(moe.moe_store_tier(st, 2)[0].tolist())

        for e in (0, 0, 0, 1):  # 0 fetched 3 times, 1 once (and more recently)
            use(e)
        use(2)  # evicts 1, the fewest fetches, though 0 was used less recently
        assert tier() == [0, 2]
        use(0)  # 0: four fetches
        assert moe.moe_store_get_stats(st)["reads"] == 3
        for e in (2, 2, 2):  # 2 now has four fetches too, and is the more recent
            use(e)
        use(4)  # a tie on fetches: the least recently used goes
        assert tier() == [2, 4]
        s = moe.moe_store_get_stats(st)
        assert s["reads"] == 4 and s["fetches"] == 10 and s["tier_hits"] == 6
    finally:
        moe.moe_store_close(st)


def test_pinned_entries_are_never_reused(expert_file):
    eb = moe.moe_expert_bytes(SHAPES)
    st = moe.moe_store_open(expert_file, SHAPES, 2, 2)
    try:
        a = moe.moe_store_fetch(st, 3, eb)
        moe.moe_store_fetch(st, 4, eb)
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_store_fetch(st, 5, eb)
        assert ei.value.status == moe.MOE_EBUSY
        # a fetch of a pinned expert pins it again and succeeds
        assert (moe.moe_store_fetch(st, 3, eb) == a).all()
        moe.moe_store_release(st, 3)
        moe.moe_store_release(st, 3)
        assert (moe.moe_store_fetch(st, 5, eb) == _region(expert_file, 5)[:eb]).all()
        assert sorted(moe.moe_store_tier(st, 2)[0]) == [4, 5]
        with pytest.raises(moe.MoeError):
            moe.moe_store_release(st, 3)  # no longer in the tier
        moe.moe_store_release(st, 4)
        moe.moe_store_release(st, 5)
    finally:
        moe.moe_store_close(st)


def test_readahead_fills_free_entries_and_keeps_unused_ones(expert_file):
    eb = moe.moe_expert_bytes(SHAPES)
    st = moe.moe_store_open(expert_file, SHAPES, 3, 2)
    try:
        assert moe.moe_store_prefetch(st, [6, 1]) == 2
        assert moe.moe_store_prefetch(st, [6]) == 0  # already there
        moe.moe_store_wait_idle(st)
        ex, state = moe.moe_store_tier(st, 3)
        assert sorted(ex[state == 2]) == [1, 6]
        # the third entry is free; a fourth expert would have to evict an
        # expert read ahead and not yet used, which readahead never does
        assert moe.moe_store_prefetch(st, [2, 3]) == 1
        moe.moe_store_wait_idle(st)
        assert (moe.moe_store_fetch(st, 6, eb) == _region(expert_file, 6)[:eb]).all()
        moe.moe_store_release(st, 6)
        s = moe.moe_store_get_stats(st)
        assert s["prefetch_reads"] == 3 and s["prefetch_used"] == 1 and s["tier_hits"] == 1
        # 6 has been used, but fetched once: 3 (never fetched) may not displace it
        assert moe.moe_store_prefetch(st, [3]) == 0
    finally:
        moe.moe_store_close(st)


def test_readahead_only_displaces_experts_fetched_no_more_often(expert_file):
    eb = moe.moe_expert_bytes(SHAPES)
    st = moe.moe_store_open(expert_file, SHAPES, 2, 1)
    try:
        def use(e):
            moe.moe_store_fetch(st, e, eb)
            moe.moe_store_release(st, e)

        def tier():
            return sorted(moe.moe_store_tier(st, 2)[0].tolist())

        for e in (0, 1, 1):  # fetches: 0 once, 1 twice
            use(e)
        assert moe.moe_store_prefetch(st, [2]) == 0  # 2 has no fetches; 0 has one
        for e in (2, 2):  # a fetch may displace 0; then 2 has two fetches
            use(e)
        assert tier() == [1, 2]
        assert moe.moe_store_prefetch(st, [0]) == 0  # 0 has one fetch, the others two
        use(0)  # 1 and 2 tie at two fetches: 1, the least recent, goes
        assert tier() == [0, 2]
        assert moe.moe_store_prefetch(st, [1]) == 1  # 1 (two fetches) may displace 2 (two)
        moe.moe_store_wait_idle(st)
        assert tier() == [0, 1]
        assert moe.moe_store_get_stats(st)["prefetch_reads"] == 1
    finally:
        moe.moe_store_close(st)


def test_open_rejects_bad_files_and_arguments(tmp_path, expert_file):
    other = synth.Shapes(512, 8, 2, 256, 512, synth.GELU_TANH)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_store_open(expert_file, other, 2, 1)
    assert ei.value.status == moe.MOE_EINVAL
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_store_open(str(tmp_path / "absent"), SHAPES, 2, 1)
    assert ei.value.status == moe.MOE_EIO
    junk = tmp_path / "junk"
    junk.write_bytes(b"\0" * 8192)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_store_open(str(junk), SHAPES, 2, 1)
    assert ei.value.status == moe.MOE_EINVAL
    short = tmp_path / "short"
    short.write_bytes(open(expert_file, "rb").read()[:-1])
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_store_open(str(short), SHAPES, 2, 1)
    assert ei.value.status == moe.MOE_EINVAL
    for slots, readers, flags in [(0, 1, 0), (9, 1, 0), (2, 0, 0), (2, 65, 0), (2, 1, 2)]:
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_store_open(expert_file, SHAPES, slots, readers, flags)
        assert ei.value.status == moe.MOE_EINVAL


@pytest.mark.parametrize("chunk", [0, 65536])
def test_read_failure_is_reported_and_retried(tmp_path, weights, chunk):
    p = str(tmp_path / "shrinks.experts")
    moe.moe_store_write(p, SHAPES, weights)
    eb = moe.moe_expert_bytes(SHAPES)
    stride = moe.moe_store_expert_stride(SHAPES)
    st = moe.moe_store_open(p, SHAPES, 2, 3)
    moe.moe_store_set_read_chunk(st, chunk)
    try:
        os.truncate(p, ALIGN + 4 * stride)  # experts 4..7 are gone
        assert (moe.moe_store_fetch(st, 3, eb) == np.fromfile(p, np.uint8)[ALIGN + 3 * stride:][:eb]).all()
        moe.moe_store_release(st, 3)
        for _ in range(2):  # the failed entry is freed; the next fetch reads again
            with pytest.raises(moe.MoeError) as ei:
                moe.moe_store_fetch(st, 6, eb)
            assert ei.value.status == moe.MOE_EIO
        s = moe.moe_store_get_stats(st)
        assert s["read_errors"] == 2 and s["reads"] == 3
        assert 6 not in moe.moe_store_tier(st, 2)[0]
    finally:
        moe.moe_store_close(st)


@pytest.mark.parametrize("chunk", [0, 4096, 65536])
def test_a_read_cut_short_inside_an_expert_fails_whole(tmp_path, weights, chunk):
    # the file ends 100 KiB into expert 2: with pieces, some of its pieces
    # land and some fail; the entry must fail as a whole, never be served
    p = str(tmp_path / "cut.experts")
    moe.moe_store_write(p, SHAPES, weights)
    eb = moe.moe_expert_bytes(SHAPES)
    stride = moe.moe_store_expert_stride(SHAPES)
    st = moe.moe_store_open(p, SHAPES, 2, 4)
    moe.moe_store_set_read_chunk(st, chunk)
    try:
        os.truncate(p, ALIGN + 2 * stride + 100 * 1024)
        assert (moe.moe_store_fetch(st, 1, eb) == np.fromfile(p, np.uint8)[ALIGN + stride:][:eb]).all()
        moe.moe_store_release(st, 1)
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_store_fetch(st, 2, eb)
        assert ei.value.status == moe.MOE_EIO
        s = moe.moe_store_get_stats(st)
        assert s["reads"] == 2 and s["read_errors"] == 1 and s["bytes_read"] == stride
    finally:
        moe.moe_store_close(st)


def test_read_chunk_must_be_page_multiple(expert_file):
    st = moe.moe_store_open(expert_file, SHAPES, 2, 1)
    try:
        for bad in (1, 4095, 6000):
            with pytest.raises(moe.MoeError) as ei:
                moe.moe_store_set_read_chunk(st, bad)
            assert ei.value.status == moe.MOE_EINVAL
        moe.moe_store_set_read_chunk(st, 10 * 2 ** 20)  # above the stride: whole-expert reads
    finally:
        moe.moe_store_close(st)


@pytest.mark.parametrize("chunk", [0, 8192])
def test_concurrent_fetches_get_their_bytes(expert_file, chunk):
    eb = moe.moe_expert_bytes(SHAPES)
    want = [_region(expert_file, e)[:eb] for e in range(SHAPES.n_experts)]
    st = moe.moe_store_open(expert_file, SHAPES, 4, 3)
    moe.moe_store_set_read_chunk(st, chunk)
    errors = []

    def worker(seed):
        rng = np.random.default_rng(seed)
        try:
            for e in rng.integers(0, SHAPES.n_experts, 40):
                got = moe.moe_store_fetch(st, int(e), eb)
                if not (got == want[e]).all():
                    errors.append(int(e))
                moe.moe_store_release(st, int(e))
        except Exception as ex:  # noqa: BLE001
            errors.append(repr(ex))

    try:
        th = [threading.Thread(target=worker, args=(i,)) for i in range(4)]
        for t in th:
            t.start()
        for t in th:
            t.join()
        assert not errors, errors
        s = moe.moe_store_get_stats(st)
        assert s["fetches"] == 160 and s["read_errors"] == 0
    finally:
        moe.moe_store_close(st)


class _TierModel:
    """The host tier's rules restated on their own: fetch counts per expert;
    a fetch takes an empty entry, else the unpinned entry whose expert has the
    fewest fetches (ties: least recently used); readahead also keeps entries
    read ahead and not yet fetched, and takes an entry only if its expert has
    no more fetches than the one read ahead. Reads finish at once here (the
    test waits for the store's readers after every request)."""

    def __init__(self, H, E):
        self.ent = [{"e": -1, "pins": 0, "used": 0, "pred": False} for _ in range(H)]
        self.freq = [0] * E
        self.tick = 0
        self.stats = dict(fetches=0, tier_hits=0, reads=0, prefetch_reads=0, prefetch_used=0)

    def _where(self, e):
        return next((i for i, x in enumerate(self.ent) if x["e"] == e), None)

    def _pick(self, ahead=None):
        for i, x in enumerate(self.ent):
            if x["e"] < 0:
                return i
        ok = [i for i, x in enumerate(self.ent) if x["pins"] == 0 and not (ahead is not None and x["pred"])]
        if not ok:
            return None
        best = min(ok, key=lambda i: (self.freq[self.ent[i]["e"]], self.ent[i]["used"]))
        if ahead is not None and self.freq[self.ent[best]["e"]] > self.freq[ahead]:
            return None
        return best

    def _assign(self, i, e, pred):
        self.tick += 1
        self.ent[i] = {"e": e, "pins": 0, "used": self.tick, "pred": pred}
        self.stats["reads"] += 1

    def fetch(self, e):
        i = self._where(e)
        hit = i is not None
        if not hit:
            i = self._pick()
            if i is None:
                return False  # every entry pinned
            self._assign(i, e, False)
        x = self.ent[i]
        self.stats["tier_hits"] += hit
        self.stats["prefetch_used"] += x["pred"]
        x["pred"] = False
        x["pins"] += 1
        self.tick += 1
        x["used"] = self.tick
        self.freq[e] += 1
        self.stats["fetches"] += 1
        return True

    def release(self, e):
        self.ent[self._where(e)]["pins"] -= 1

    def prefetch(self, experts):
        q = 0
        for e in experts:
            if self._where(e) is not None:
                continue
            i = self._pick(ahead=e)
            if i is None:
                continue
            self._assign(i, e, True)
            q += 1
        self.stats["prefetch_reads"] += q
        return q


@pytest.mark.parametrize("seed,chunk", [(0, 0), (1, 0), (2, 65536), (3, 16384)])
def test_tier_follows_its_rules_on_random_requests(expert_file, seed, chunk):
    H, E = 3, SHAPES.n_experts
    eb = moe.moe_expert_bytes(SHAPES)
    want = [_region(expert_file, e)[:eb] for e in range(E)]
    rng = np.random.default_rng(seed)
    st = moe.moe_store_open(expert_file, SHAPES, H, 2)
    moe.moe_store_set_read_chunk(st, chunk)
    model = _TierModel(H, E)
    held = []
    try:
        for step in range(300):
            op = rng.random()
            if op < 0.45:
                e = int(rng.integers(0, E))
                ok = model.fetch(e)
                try:
                    got = moe.moe_store_fetch(st, e, eb)
                    assert ok and (got == want[e]).all(), (step, e)
                    held.append(e)
                except moe.MoeError as ex:
                    assert not ok and ex.status == moe.MOE_EBUSY, (step, e)
            elif op < 0.8 and held:
                e = held.pop(int(rng.integers(0, len(held))))
                model.release(e)
                moe.moe_store_release(st, e)
            else:
                ask = [int(v) for v in rng.integers(0, E, int(rng.integers(1, 4)))]
                assert moe.moe_store_prefetch(st, ask) == model.prefetch(ask), (step, ask)
                moe.moe_store_wait_idle(st)
            ex, state = moe.moe_store_tier(st, H)
            assert ex.tolist() == [x["e"] for x in model.ent], (step, ex, model.ent)
            assert all(s in (0, 2) for s in state.tolist())
            got = moe.moe_store_get_stats(st)
            assert {k: got[k] for k in model.stats} == model.stats, step
        for e in held:
            moe.moe_store_release(st, e)
    finally:
        moe.moe_store_close(st)
