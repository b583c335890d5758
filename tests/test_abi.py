"""Host-side checks of libmoe.so that need no GPU: the library loads, exports
every function include/moe.h declares, and rejects bad arguments with a status
before anything is enqueued (no CUDA call is made on these paths)."""
import ctypes
import os
import re

import pytest

import sparse_mixture_experts_64_b300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    for m in re.finditer(r"^\s*(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", src, flags=re.M):
        names.append(m.group(1))
    return sorted(set(names))


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert set(moe.EXPORTED) <= set(names) and len(names) >= 11
    lib = ctypes.CDLL(moe.library_path())
    for n in names:
        assert hasattr(lib, n), n


def _cfg(**kw):
    base = dict(T=64, d=128, N=8, k=2, h=256, dtype="bf16")
    base.update(kw)
    return moe.make_config(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(T=0), moe.MOE_ERR_INVALID_ARG),
    (dict(T=65537), moe.MOE_ERR_INVALID_ARG),
    (dict(N=0), moe.MOE_ERR_INVALID_ARG),
    (dict(N=257, k=2), moe.MOE_ERR_INVALID_ARG),
    (dict(k=0), moe.MOE_ERR_INVALID_ARG),
    (dict(k=9, N=16), moe.MOE_ERR_INVALID_ARG),
    (dict(k=3, N=2), moe.MOE_ERR_INVALID_ARG),
    (dict(d=96), moe.MOE_ERR_UNSUPPORTED),            # bf16 needs multiples of 64
    (dict(h=100), moe.MOE_ERR_UNSUPPORTED),
    (dict(h_shared=32), moe.MOE_ERR_UNSUPPORTED),
    (dict(d=12, dtype="f32"), moe.MOE_ERR_UNSUPPORTED),  # fp32 needs multiples of 8
    (dict(capacity_factor=(1, 0)), moe.MOE_ERR_INVALID_ARG),
    (dict(dtype=7), moe.MOE_ERR_INVALID_ARG),
    (dict(gating=5), moe.MOE_ERR_INVALID_ARG),
    (dict(act=3), moe.MOE_ERR_INVALID_ARG),
])
def test_config_validation(kw, status):
    c = _cfg(**kw)
    assert moe.moe_validate_config(c) == status
    assert moe.moe_workspace_size(c) == 0


def test_valid_configs_and_sizes():
    c = _cfg()
    assert moe.moe_validate_config(c) == moe.MOE_OK
    assert moe.moe_workspace_size(c) > 0
    assert moe.moe_max_rows(c) == 64 * 2
    assert moe.moe_capacity(c) == 0
    sw = moe.make_config(T=4096, d=768, N=8, k=1, h=3072, act="relu", gating="softmax_then_topk",
                         capacity_factor=(5, 4), router_bias=True)
    assert moe.moe_capacity(sw) == 640
    assert moe.moe_max_rows(sw) == 4096
    sw2 = moe.make_config(T=4096, d=768, N=8, k=2, h=3072, capacity_factor=(1, 2))
    assert moe.moe_capacity(sw2) == 256 and moe.moe_max_rows(sw2) == 8 * 256
    # the router calls need only the leading part of the workspace
    assert 0 < moe.moe_router_workspace_size(c) < moe.moe_workspace_size(c)
    ds = moe.make_config(T=8192, d=7168, N=256, k=8, h=2048, h_shared=2048, gating="softmax_then_topk")
    assert moe.moe_router_workspace_size(ds) <= 32 << 20
    ec = moe.make_config(T=64, d=128, N=8, k=2, h=256, capacity_factor=(2, 1), routing="expert_choice")
    assert moe.moe_router_workspace_size(ec) == 0
    assert moe.moe_router_workspace_size(_cfg(T=0)) == 0
    tiny = moe.make_config(T=256, d=64, N=4, k=2, h=128, dtype="f32")
    assert moe.moe_validate_config(tiny) == moe.MOE_OK
    assert moe.status_str(moe.MOE_ERR_TIMEOUT) == "MOE_ERR_TIMEOUT"


NONE = ctypes.c_size_t(-1).value


def test_kept_preactivation_regions():
    """save_preact adds the pre-activation regions to the workspace (bf16, dispatch
    order) and only where moe_forward keeps them."""
    kw = dict(T=8192, d=7168, N=256, k=8, h=2048, h_shared=2048, gating="softmax_then_topk")
    plain, keep = moe.make_config(**kw), moe.make_config(**kw, save_preact=True)
    assert moe.moe_preact_offset(plain) == NONE
    rmax = moe.moe_max_rows(keep)
    grow = moe.moe_workspace_size(keep) - moe.moe_workspace_size(plain)
    need = rmax * 2 * 2048 * 2 + 8192 * 2 * 2048 * 2
    assert need - 512 <= grow <= need  # (an empty region still takes 256 bytes)
    off, off_sh = moe.moe_preact_offset(keep), moe.moe_preact_offset(keep, shared=True)
    assert off % 256 == 0 and off_sh >= off + rmax * 2 * 2048 * 2
    assert off_sh + 8192 * 2 * 2048 * 2 <= moe.moe_workspace_size(keep)
    # the router's prefix and the backward scratch (which then holds no pre-activations)
    assert moe.moe_router_workspace_size(keep) == moe.moe_router_workspace_size(plain)
    bws = lambda c: moe._lib.moe_backward_workspace_size(ctypes.byref(c))  # noqa: E731
    assert (bws(plain) - bws(keep)
            >= need - 512)
    # ReLU experts keep X W1ᵀ only; no shared expert, no shared region
    relu = moe.make_config(T=4096, d=768, N=8, k=1, h=3072, act="relu", save_preact=True)
    assert moe.moe_preact_offset(relu) != NONE and moe.moe_preact_offset(relu, shared=True) == NONE
    # nothing is kept on the fp32, forced CUDA-core, weights-as-M and Expert Choice paths
    for c in (moe.make_config(T=256, d=64, N=4, k=2, h=128, dtype="f32", save_preact=True),
              moe.make_config(**kw, save_preact=True, debug_flags=moe.MOE_DEBUG_FORCE_SIMT_FFN),
              moe.make_config(**kw, save_preact=True, debug_flags=moe.MOE_DEBUG_FFN_SWAP),
              moe.make_config(T=64, d=128, N=8, k=2, h=256, capacity_factor=(2, 1),
                              routing="expert_choice", save_preact=True)):
        assert moe.moe_validate_config(c) == moe.MOE_OK
        assert moe.moe_preact_offset(c) == NONE
    bad = moe.make_config(**kw)
    bad.save_preact = 2
    assert moe.moe_validate_config(bad) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_preact_offset(bad) == NONE


FAKE = 1 << 20          # a 256-aligned address that is never dereferenced on these paths


def _raw(fn, *args):
    return getattr(moe._lib, fn)(*args)


def test_null_pointers_rejected_before_launch():
    c = _cfg()
    cp = ctypes.byref(c)
    ws = moe.moe_workspace_size(c)
    # forward: x missing
    st = _raw("moe_forward", cp, None, FAKE, None, FAKE, FAKE, FAKE, None, None, None, FAKE,
              None, None, None, None, None, FAKE, ws, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    # forward: gated experts need w_up
    st = _raw("moe_forward", cp, FAKE, FAKE, None, FAKE, None, FAKE, None, None, None, FAKE,
              None, None, None, None, None, FAKE, ws, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    # router: bias declared but missing
    cb = _cfg(router_bias=True)
    st = _raw("moe_router_topk", ctypes.byref(cb), FAKE, FAKE, None, FAKE, FAKE, None, None,
              FAKE, FAKE, FAKE, None, FAKE, moe.moe_workspace_size(cb), None)
    assert st == moe.MOE_ERR_INVALID_ARG
    # combine: shared expert declared but weights missing
    cs = _cfg(h_shared=128)
    st = _raw("moe_combine", ctypes.byref(cs), FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE,
              FAKE, moe.moe_workspace_size(cs), None)
    assert st == moe.MOE_ERR_INVALID_ARG
    # misaligned activation pointer
    st = _raw("moe_dispatch", cp, FAKE + 2, FAKE, FAKE, FAKE, None, 0, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    # training router: a non-finite noise weight with noise, a missing output
    for wn in (float("nan"), float("inf")):
        st = _raw("moe_router_topk_train", cp, FAKE, FAKE, None, FAKE, wn, FAKE, FAKE, None, None,
                  FAKE, FAKE, FAKE, None, None, FAKE, ws, None)
        assert st == moe.MOE_ERR_INVALID_ARG
    st = _raw("moe_router_topk_train", cp, FAKE, FAKE, None, None, 0.0, None, FAKE, None, None,
              FAKE, FAKE, FAKE, None, FAKE, FAKE, ws, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    # sharded router: the shard's config carries no capacity (it is global), slot
    # counts and bases are required, global_T covers at least this shard, aux needs
    # the global sums
    ccap = _cfg(capacity_factor=(1, 1))
    st = _raw("moe_router_shard_stats", ctypes.byref(ccap), FAKE, FAKE, None, FAKE, FAKE, FAKE, None,
              FAKE, moe.moe_workspace_size(ccap), None)
    assert st == moe.MOE_ERR_INVALID_ARG
    st = _raw("moe_router_shard_stats", cp, FAKE, FAKE, None, FAKE, FAKE, None, None, FAKE, ws, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    st = _raw("moe_router_shard_assign", cp, FAKE, None, 0, None, None, c.T, None, FAKE, FAKE, FAKE,
              None, FAKE, ws, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    st = _raw("moe_router_shard_assign", cp, FAKE, FAKE, 0, None, None, c.T - 1, None, FAKE, FAKE,
              FAKE, None, FAKE, ws, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    st = _raw("moe_router_shard_assign", cp, FAKE, FAKE, 0, None, None, c.T, None, FAKE, FAKE, FAKE,
              FAKE, FAKE, ws, None)
    assert st == moe.MOE_ERR_INVALID_ARG


def test_expert_choice_config_rules():
    """Expert Choice needs a capacity factor and T <= 16384; its rows are N * min(C, T);
    the token-choice calls refuse it and its forward takes no token-choice outputs."""
    assert moe.moe_validate_config(_cfg(routing="expert_choice")) == moe.MOE_ERR_INVALID_ARG
    ec = _cfg(routing="expert_choice", capacity_factor=(2, 1))
    assert moe.moe_validate_config(ec) == moe.MOE_OK
    assert moe.moe_max_rows(ec) == 8 * 16                            # N * ceil(64 * 2 / 8)
    big = _cfg(routing="expert_choice", capacity_factor=(1, 1), T=16385)
    assert moe.moe_validate_config(big) == moe.MOE_ERR_UNSUPPORTED
    whole = _cfg(routing="expert_choice", capacity_factor=(64, 1))  # C >= T: every token
    assert moe.moe_max_rows(whole) == 8 * 64
    bad = _cfg(routing=7)
    assert moe.moe_validate_config(bad) == moe.MOE_ERR_INVALID_ARG
    cp = ctypes.byref(ec)
    ws = moe.moe_workspace_size(ec)
    assert _raw("moe_router_topk", cp, FAKE, FAKE, None, FAKE, FAKE, None, None, FAKE, FAKE, FAKE,
                None, FAKE, ws, None) == moe.MOE_ERR_UNSUPPORTED
    assert _raw("moe_combine", cp, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE, FAKE, ws,
                None) == moe.MOE_ERR_UNSUPPORTED
    assert _raw("moe_router_topk_noalloc", cp, FAKE, FAKE, None, FAKE, FAKE, None, None, FAKE,
                FAKE, FAKE, None, None) == moe.MOE_ERR_UNSUPPORTED
    tc = _cfg()
    assert _raw("moe_router_expert_choice", ctypes.byref(tc), FAKE, FAKE, None, FAKE, FAKE, FAKE,
                FAKE, FAKE, FAKE, moe.moe_workspace_size(tc), None) == moe.MOE_ERR_UNSUPPORTED
    # forward with a token-choice output pointer
    st = _raw("moe_forward", cp, FAKE, FAKE, None, FAKE, FAKE, FAKE, None, None, None, FAKE,
              FAKE, None, None, None, None, FAKE, ws, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    # missing list outputs
    assert _raw("moe_router_expert_choice", cp, FAKE, FAKE, None, FAKE, FAKE, FAKE, None, FAKE,
                FAKE, ws, None) == moe.MOE_ERR_INVALID_ARG


def test_workspace_checks_before_launch():
    c = _cfg()
    cp = ctypes.byref(c)
    ws = moe.moe_workspace_size(c)
    args = [FAKE, FAKE, None, FAKE, FAKE, FAKE, None, None, None, FAKE, None, None, None, None,
            None]
    assert _raw("moe_forward", cp, *args, None, ws, None) == moe.MOE_ERR_WORKSPACE
    assert _raw("moe_forward", cp, *args, FAKE, ws - 1, None) == moe.MOE_ERR_WORKSPACE
    assert _raw("moe_forward", cp, *args, FAKE + 16, ws, None) == moe.MOE_ERR_WORKSPACE
    assert _raw("moe_router_topk", cp, FAKE, FAKE, None, FAKE, FAKE, None, None, FAKE, FAKE, FAKE,
                None, FAKE, 16, None) == moe.MOE_ERR_WORKSPACE
    assert _raw("moe_router_topk_train", cp, FAKE, FAKE, None, None, 0.0, FAKE, FAKE, None, None,
                FAKE, FAKE, FAKE, None, FAKE, FAKE, 16, None) == moe.MOE_ERR_WORKSPACE
    assert _raw("moe_check_error", None, None) == moe.MOE_ERR_WORKSPACE


def test_product_path_has_no_cpu_fallback():
    """The binding only marshals arguments: it imports nothing from the oracle."""
    import inspect
    src = inspect.getsource(moe)
    assert "oracle" not in src.replace("no Python or CPU fallback", "")
    pkg = os.path.dirname(moe.__file__)
    for name in os.listdir(pkg):
        if name.endswith(".py"):
            with open(os.path.join(pkg, name)) as f:
                assert "import oracle" not in f.read() and "from oracle" not in open(
                    os.path.join(pkg, name)).read()


def test_forward_graph_checks_before_capture():
    """moe_forward_graph_create returns its status before any stream or capture exists
    when the handle, the events, the config or the workspace is wrong; destroying a
    NULL graph is a no-op and launching one is an error."""
    lib = ctypes.CDLL(moe.library_path())
    lib.moe_forward_graph_create.restype = ctypes.c_int32
    P = ctypes.c_void_p
    out = P()
    good = _cfg()

    def create(cfg, ws=0x1000, ws_bytes=1 << 40, events=None, n_events=0, out_p=ctypes.byref(out)):
        args = [ctypes.byref(cfg)] + [P(0x100)] * 15 + [P(ws), ctypes.c_size_t(ws_bytes), events,
                                                         ctypes.c_int32(n_events), out_p]
        return lib.moe_forward_graph_create(*args)

    assert create(good, out_p=None) == moe.MOE_ERR_INVALID_ARG
    assert create(good, n_events=6) == moe.MOE_ERR_INVALID_ARG               # NULL events
    three = (P * 3)(1, 2, 3)
    assert create(good, events=three, n_events=3) == moe.MOE_ERR_INVALID_ARG
    assert create(_cfg(T=0)) == moe.MOE_ERR_INVALID_ARG
    assert create(_cfg(d=96)) == moe.MOE_ERR_UNSUPPORTED
    assert create(good, ws=0) == moe.MOE_ERR_WORKSPACE
    assert create(good, ws_bytes=16) == moe.MOE_ERR_WORKSPACE
    assert out.value is None
    assert lib.moe_forward_graph_destroy(None) == moe.MOE_OK
    assert lib.moe_forward_graph_launch(None, None) == moe.MOE_ERR_INVALID_ARG
