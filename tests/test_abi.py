"""The C-ABI library without a GPU: it loads, exports every declared entry
point, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_layout.h")


@pytest.fixture(scope="module")
def moe():
    from combine_moe_layout_04_gb300 import _build
    _build.build()
    import combine_moe_layout_04_gb300 as m
    m.load_library()
    return m


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(moe_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("moe_workspace_bytes", "moe_layout", "moe_stats_words", "moe_stats", "moe_dispatch",
              "moe_combine", "moe_status", "moe_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(moe):
    lib = ctypes.CDLL(moe.LIB_PATH)
    for n in _declared():
        assert hasattr(lib, n), n
    assert set(moe.EXPORTED) <= set(_declared())


def test_status_strings(moe):
    assert moe.moe_status_string(0) == "ok"
    assert "misaligned" in moe.moe_status_string(moe.MOE_ERR_ALIGN)
    assert moe.moe_status_string(1234) == "unknown status"


def _p(moe, **kw):
    base = dict(num_tokens=256, hidden=1024, topk=2, num_experts=16, num_ranks=4, ranks_per_host=2,
                num_src_ranks=4, dtype=moe.MOE_DTYPE_BF16)
    base.update(kw)
    return moe.Problem(**base)


@pytest.mark.parametrize("bad", [
    dict(topk=0), dict(topk=33), dict(num_experts=1025), dict(num_ranks=3, ranks_per_host=2),
    dict(num_ranks=1024, ranks_per_host=8), dict(num_src_ranks=5), dict(num_experts=18),
    dict(num_tokens=250), dict(hidden=1020), dict(dtype=1, hidden=1000), dict(dtype=7),
    dict(num_tokens=1 << 28, topk=8, num_src_ranks=1), dict(num_tokens=-1),
    dict(hidden=(1 << 20) + 8), dict(hidden=1 << 30), dict(dtype=1, hidden=(1 << 20) + 128)])
def test_host_rejects_bad_problems(moe, bad):
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_workspace_bytes(_p(moe, **bad))
    assert ei.value.code == moe.MOE_ERR_INVALID
    assert moe.moe_stats_words(_p(moe, **bad)) == 0


def test_workspace_and_stats_sizes(moe):
    p = _p(moe)
    n = moe.moe_workspace_bytes(p)
    assert n % 256 == 0 and 0 < n < 1 << 20
    assert moe.moe_stats_words(p) == 32 + 9 * 4 + 6 * 4
    big = _p(moe, num_tokens=16384, hidden=7168, topk=8, num_experts=128, num_ranks=16,
             ranks_per_host=8, num_src_ranks=1, dtype=moe.MOE_DTYPE_FP8_E4M3)
    assert moe.moe_workspace_bytes(big) < 1 << 20


class _Fake:
    """A pointer-shaped stand-in: the host checks below must reject the call
    from the address alone, before any device access."""
    def __init__(self, addr):
        self.addr = addr

    def data_ptr(self):
        return self.addr


def test_host_rejects_misaligned_rows(moe):
    p = _p(moe)
    lay = moe.Layout.__new__(moe.Layout)
    for n in moe._LAYOUT_FIELDS:
        setattr(lay, n, _Fake(0x10000))
    good, odd = _Fake(0x20000), _Fake(0x20008)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_dispatch(p, lay, odd, None, good, None, stream=0)
    assert ei.value.code == moe.MOE_ERR_ALIGN
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_combine(p, lay, good, _Fake(0x30000), odd, stream=0)
    assert ei.value.code == moe.MOE_ERR_ALIGN
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layout(p, _Fake(0x40000), _Fake(0x50010), lay, stream=0)
    assert ei.value.code == moe.MOE_ERR_ALIGN
    pf = _p(moe, dtype=moe.MOE_DTYPE_FP8_E4M3)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_dispatch(pf, lay, good, None, good, None, stream=0)   # fp8 needs scales
    assert ei.value.code == moe.MOE_ERR_INVALID


def test_host_rejects_bad_relay_calls(moe):
    """Relay entry points: NULL arrays, negative capacity and misaligned rows
    are rejected on the host."""
    p = _p(moe)
    lay = moe.Layout.__new__(moe.Layout)
    for n in moe._LAYOUT_FIELDS:
        setattr(lay, n, _Fake(0x10000))
    rel = moe.Relay.__new__(moe.Relay)
    rel.relay_pos, rel.relay_src, rel.slot_relay, rel.capacity = _Fake(0x60000), _Fake(0x61000), _Fake(0x62000), 512
    good, odd = _Fake(0x20000), _Fake(0x20008)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_relay_layout(p, lay, _Fake(0x50010), rel, stream=0)      # workspace not 256-aligned
    assert ei.value.code == moe.MOE_ERR_ALIGN
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_dispatch_relay(p, lay, rel, good, None, odd, None, good, None, stream=0)
    assert ei.value.code == moe.MOE_ERR_ALIGN
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_combine_relay(p, lay, rel, good, _Fake(0x30000), good, odd, stream=0)
    assert ei.value.code == moe.MOE_ERR_ALIGN
    rel.capacity = -1
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_combine_relay(p, lay, rel, good, _Fake(0x30000), good, good, stream=0)
    assert ei.value.code == moe.MOE_ERR_INVALID
    rel.capacity, rel.slot_relay = 512, _Fake(0)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_dispatch_relay(p, lay, rel, good, None, good, None, good, None, stream=0)
    assert ei.value.code == moe.MOE_ERR_INVALID


def test_host_rejects_bad_group_calls(moe):
    p = _p(moe)
    lay = moe.Layout.__new__(moe.Layout)
    for n in moe._LAYOUT_FIELDS:
        setattr(lay, n, _Fake(0x10000))
    good, odd, ids, grp = _Fake(0x20000), _Fake(0x20008), _Fake(0x70000), _Fake(0x71000)
    for bad_g in (0, moe.MOE_MAX_GROUPS + 1):
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_expert_groups(p, bad_g, grp, stream=0)
        assert ei.value.code == moe.MOE_ERR_INVALID
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_combine_group(p, lay, ids, grp, 2, 2, good, _Fake(0x30000), good, good, stream=0)  # group >= G
    assert ei.value.code == moe.MOE_ERR_INVALID
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_combine_group(p, lay, ids, grp, 0, 2, good, _Fake(0x30000), None, good, stream=0)  # acc needed
    assert ei.value.code == moe.MOE_ERR_INVALID
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_combine_group(p, lay, ids, grp, 0, 2, good, _Fake(0x30000), odd, good, stream=0)
    assert ei.value.code == moe.MOE_ERR_ALIGN
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_dispatch_group(p, lay, ids, grp, 0, odd, None, good, None, stream=0)
    assert ei.value.code == moe.MOE_ERR_ALIGN


def test_stats_call_shapes():
    """moe_stats hands a host record over and synchronises; moe_stats_device
    is the asynchronous device copy (the header says which is which)."""
    text = open(HEADER).read()
    flat = re.sub(r"\s+", " ", text)
    assert ("int moe_stats(const moe_problem* problem, const moe_layout_t* layout, "
            "const void* workspace, int64_t* host_stats, moe_stream_t stream);") in flat
    assert ("int moe_stats_device(const moe_problem* problem, const void* workspace, int64_t* device_stats, "
            "moe_stream_t stream);") in flat
    decl = flat[flat.index("/* Statistics of a layout, copied to HOST memory"):flat.index("int moe_stats(")]
    assert "synchronises the stream" in decl


def test_every_call_cites_its_passage():
    """Each exported call's declaration comment names the page that defines
    it, or says that the pages have no counterpart."""
    text = open(HEADER).read()
    pages = ("Balancing and Beyond", "Poor HybridEP", "Profiling when rank unbalance", "no counterpart")
    cited_elsewhere = {"moe_stats_words", "moe_status_string"}   # sizes and names, no operation
    for name in _declared():
        if name in cited_elsewhere:
            continue
        at = re.search(r"^\s*int " + name + r"\(", text, flags=re.M).start()
        comment = text[text.rindex("/*", 0, at):at]
        assert any(p in comment for p in pages), name


def test_host_stats_rejected_on_host(moe):
    p = _p(moe)
    lay = moe.Layout.__new__(moe.Layout)
    for n in moe._LAYOUT_FIELDS:
        setattr(lay, n, _Fake(0x10000))
    lay.stats = None
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_stats(p, lay, None, stream=0)           # neither layout.stats nor a workspace
    assert ei.value.code == moe.MOE_ERR_INVALID
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_stats(p, lay, _Fake(0x50010), stream=0)  # workspace not 256-byte aligned
    assert ei.value.code == moe.MOE_ERR_ALIGN
    lay.stats = _Fake(0x40004)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_stats(p, lay, None, stream=0)            # device record not 8-byte aligned
    assert ei.value.code == moe.MOE_ERR_ALIGN
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_stats_device(p, _Fake(0x50000), _Fake(0x40004), stream=0)
    assert ei.value.code == moe.MOE_ERR_ALIGN


def test_tuning_checked_on_host(moe):
    """moe_tuning (launch shapes of the layout and the movers): every out-of-range field is
    rejected by every call before anything is enqueued; defaults pass."""
    import ctypes
    p = _p(moe)
    base = moe.moe_workspace_bytes(p)
    for good in (dict(), dict(dispatch_kind=moe.MOE_MOVE_BULK, dispatch_warps=16, dispatch_stages=3,
                              dispatch_chunk_bytes=4096),
                 dict(dispatch_kind=moe.MOE_MOVE_VECTOR, dispatch_sms=1, dispatch_ctas_per_sm=8),
                 dict(combine_kind=moe.MOE_MOVE_VECTOR, combine_sms=152, combine_ctas_per_sm=3),
                 dict(layout_kind=moe.MOE_LAYOUT_SPLIT), dict(layout_kind=moe.MOE_LAYOUT_TWO_KERNELS)):
        p.tuning = moe.Tuning(**good)
        assert moe.moe_workspace_bytes(p) == base
    for bad in (dict(dispatch_kind=3), dict(combine_kind=-1), dict(dispatch_sms=-1), dict(combine_sms=-4),
                dict(dispatch_ctas_per_sm=9), dict(dispatch_warps=17), dict(dispatch_stages=9),
                dict(dispatch_chunk_bytes=100), dict(dispatch_chunk_bytes=1000), dict(dispatch_chunk_bytes=32784),
                dict(dispatch_warps=16, dispatch_stages=8, dispatch_chunk_bytes=7168), dict(combine_ctas_per_sm=4),
                dict(layout_kind=4), dict(layout_kind=-1)):
        p.tuning = moe.Tuning(**bad)
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_workspace_bytes(p)
        assert ei.value.code == moe.MOE_ERR_INVALID, bad
    # reserved words must stay zero
    p.tuning = moe.Tuning()
    pc = p.c()
    pc._tuning.reserved[3] = 1
    n = ctypes.c_size_t(0)
    assert moe.load_library().moe_workspace_bytes(ctypes.byref(pc), ctypes.byref(n)) == moe.MOE_ERR_INVALID


def test_tuning_from_environment(moe):
    t = moe.Tuning.from_env({"MOE_DISPATCH_KIND": "bulk", "MOE_DISPATCH_WARPS": "6", "MOE_COMBINE_SMS": "76",
                             "MOE_COMBINE_KIND": "vector", "UNRELATED": "1"})
    assert t.dispatch_kind == moe.MOE_MOVE_BULK and t.dispatch_warps == 6
    assert t.combine_kind == moe.MOE_MOVE_VECTOR and t.combine_sms == 76 and t.dispatch_sms == 0
    assert t.layout_kind == moe.MOE_LAYOUT_AUTO
    for name, kind in (("split", moe.MOE_LAYOUT_SPLIT), ("FUSED", moe.MOE_LAYOUT_FUSED),
                       ("two_kernels", moe.MOE_LAYOUT_TWO_KERNELS), ("2", moe.MOE_LAYOUT_FUSED)):
        assert moe.Tuning.from_env({"MOE_LAYOUT_KIND": name}).layout_kind == kind
