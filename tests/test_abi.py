"""Host-side checks of the C ABI (no GPU needed): the library builds, loads and
exports every function include/moe.h declares; argument validation rejects bad
calls before anything is enqueued; host helpers (capacity rule, routing-map
bytes, buffer ring) behave as documented."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__

    __graft_entry__.build_library()
    import permute_grouped_expert_gb300 as m

    return m


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w[\w\s\*]*?\b(moe_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(moe):
    names = declared_functions()
    assert len(names) >= 16, names
    lib = ctypes.CDLL(moe.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(moe.exported_symbols())


def test_binding_constants_match_the_header(moe):
    """The Python binding's status, dtype and format constants equal the header's."""
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    defines = dict((k, int(v)) for k, v in re.findall(r"#define\s+MOE_(DEV_ERR_\w+)\s+(\d+)", text))
    assert defines, "no device status bits found in moe.h"
    for k, v in defines.items():
        assert getattr(moe, k) == v, k
    enums = dict((k, int(v)) for k, v in re.findall(r"\b(MOE_(?:ERR|OK|DTYPE|COMBINE|ROUTING)\w*)\s*=\s*(\d+)", text))
    checked = 0
    for k, v in enums.items():
        name = k[4:] if k.startswith("MOE_DTYPE") or k.startswith("MOE_COMBINE") or k.startswith("MOE_ROUTING") else k
        if hasattr(moe, name):
            assert getattr(moe, name) == v, name
            checked += 1
    assert checked == len(enums), (checked, len(enums))


def test_capacity_rule_golden(moe):
    path = os.path.join(ROOT, "tests", "golden", "capacity.txt")
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        rows, factor, align, cap = line.split()
        assert moe.moe_capacity(int(rows), float(factor), int(align)) == int(cap)
    with pytest.raises(moe.MoeError):
        moe.moe_capacity(-1, 1.5, 4)
    with pytest.raises(moe.MoeError):
        moe.moe_capacity(10, 0.0, 4)


def test_routing_map_bytes_golden(moe):
    path = os.path.join(ROOT, "tests", "golden", "routing_bytes.txt")
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        layout, T, E, K, nbytes = line.split()
        fmt = moe.ROUTING_SPARSE_BOOL if layout == "sparse" else moe.ROUTING_DENSE_I16
        assert moe.moe_routing_map_bytes(fmt, int(T), int(E), int(K)) == int(nbytes)


def test_workspace_queries(moe):
    s = moe.Shape(T=8192, H=7168, E=32, K=8, I=2048)
    assert moe.moe_preprocess_workspace_size(s) > 8192 * 8 * 2
    lay = moe.Layout(32, 70000)
    assert moe.moe_grouped_mlp_workspace_size(s, lay, moe.DTYPE_BF16) >= 70000 * 2048 * 2
    with pytest.raises(moe.MoeError):
        moe.moe_preprocess_workspace_size(moe.Shape(T=8, H=128, E=2000, K=2))
    with pytest.raises(moe.MoeError):
        moe.moe_grouped_mlp_workspace_size(moe.Shape(T=8, H=128, E=4, K=2, I=100), lay, moe.DTYPE_BF16)


def test_grouped_mlp_kernel_count(moe):
    """bf16 on single SMs is one fused FC1 + FC2 kernel; SM pairs (>= 4096
    capacity rows per expert), FP8 and NVFP4 launch FC1 and FC2 separately."""
    s = moe.Shape(T=4096, H=2048, E=64, K=8, I=1024)
    assert moe.moe_grouped_mlp_kernel_count(s, moe.Layout(128, 49152), moe.DTYPE_BF16) == 1
    assert moe.moe_grouped_mlp_kernel_count(s, moe.Layout(128, 4096 * 64), moe.DTYPE_BF16) == 2
    assert moe.moe_grouped_mlp_kernel_count(s, moe.Layout(128, 4095 * 64), moe.DTYPE_BF16) == 1
    assert moe.moe_grouped_mlp_kernel_count(s, moe.Layout(128, 49152), moe.DTYPE_FP8_E4M3_B128) == 2
    assert moe.moe_grouped_mlp_kernel_count(s, moe.Layout(128, 49152), moe.DTYPE_NVFP4) == 2
    assert moe.moe_grouped_mlp_kernel_count(s, moe.Layout(128, 0), moe.DTYPE_BF16) == 0
    with pytest.raises(moe.MoeError):
        moe.moe_grouped_mlp_kernel_count(s, moe.Layout(128, 49152), 7)


def _c_call(moe, fn, *args):
    return getattr(moe.library(), fn)(*args)


def test_shape_and_layout_limits(moe):
    """The documented limits of moe_shape / moe_layout are enforced before any
    launch: 1 <= E <= 1024, 1 <= K <= min(E, 128), T >= 0, T*K and the padded
    total below 2^31, capacity below 2^31, pad multiple >= 1."""
    fake = ctypes.c_void_p(0x1000)
    routing = moe._Routing(0, fake, None)
    handle = moe._HandleDev(*([fake] * 8))
    lib = moe.library()
    byref = ctypes.byref

    def pre(shape, layout):
        return lib.moe_preprocess(byref(routing), byref(shape), byref(layout), byref(handle), fake, 1 << 40, None)

    ok_layout = moe._Layout(32, 1024)
    bad_shapes = [moe._Shape(64, 256, 0, 1, 0), moe._Shape(64, 256, 1025, 8, 0), moe._Shape(64, 256, 256, 129, 0),
                  moe._Shape(64, 256, 4, 8, 0), moe._Shape(-1, 256, 8, 2, 0), moe._Shape(1 << 26, 256, 256, 32, 0),
                  moe._Shape(64, 256, 8, 0, 0)]
    for sh in bad_shapes:
        assert pre(sh, ok_layout) == moe.MOE_ERR_INVALID_ARG, (sh.T, sh.E, sh.K)
    good = moe._Shape(64, 256, 8, 2, 0)
    for lay in [moe._Layout(0, 1024), moe._Layout(32, -1), moe._Layout(32, 1 << 31), moe._Layout(1 << 28, 1024)]:
        assert pre(good, lay) == moe.MOE_ERR_INVALID_ARG, (lay.pad_multiple, lay.capacity)


def test_validation_rejects_before_any_launch(moe):
    """Bad arguments return MOE_ERR_INVALID_ARG without touching the GPU
    (these pointers are never dereferenced)."""
    fake = ctypes.c_void_p(0x1000)
    good_shape = moe._Shape(64, 256, 8, 2, 128)
    good_layout = moe._Layout(32, 1024)
    routing = moe._Routing(0, fake, None)
    handle = moe._HandleDev(*([fake] * 8))
    h_missing = moe._HandleDev(*([fake] * 7 + [None]))
    byref = ctypes.byref
    lib = moe.library()
    # null routing map
    assert lib.moe_preprocess(byref(moe._Routing(0, None, None)), byref(good_shape), byref(good_layout),
                              byref(handle), fake, 1 << 30, None) == moe.MOE_ERR_INVALID_ARG
    # bad routing format
    assert lib.moe_preprocess(byref(moe._Routing(7, fake, None)), byref(good_shape), byref(good_layout),
                              byref(handle), fake, 1 << 30, None) == moe.MOE_ERR_INVALID_ARG
    # K > E
    assert lib.moe_preprocess(byref(routing), byref(moe._Shape(64, 256, 2, 4, 0)), byref(good_layout),
                              byref(handle), fake, 1 << 30, None) == moe.MOE_ERR_INVALID_ARG
    # negative capacity / zero pad multiple
    assert lib.moe_preprocess(byref(routing), byref(good_shape), byref(moe._Layout(32, -1)), byref(handle), fake,
                              1 << 30, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_preprocess(byref(routing), byref(good_shape), byref(moe._Layout(0, 10)), byref(handle), fake,
                              1 << 30, None) == moe.MOE_ERR_INVALID_ARG
    # a pad multiple whose largest padded total T*K + E*(m-1) does not fit int32 row ids
    assert lib.moe_preprocess(byref(routing), byref(good_shape), byref(moe._Layout(1 << 28, 1024)), byref(handle),
                              fake, 1 << 30, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_preprocess(byref(routing), byref(good_shape), byref(moe._Layout(1 << 40, 1024)), byref(handle),
                              fake, 1 << 30, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_permute(byref(handle), byref(good_shape), byref(moe._Layout(1 << 28, 1024)),
                                    moe.DTYPE_BF16, fake, None, byref(routing), fake, None, None,
                                    None) == moe.MOE_ERR_INVALID_ARG
    # the same checks come before the size rule of the allocation-free entry point
    assert lib.moe_preprocess_noalloc(byref(routing), byref(moe._Shape(1 << 22, 128, 64, 8, 0)),
                                      byref(moe._Layout(0, 1024)), byref(handle), None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_preprocess_noalloc(byref(routing), byref(good_shape), byref(good_layout), byref(h_missing),
                                      None) == moe.MOE_ERR_INVALID_ARG
    # workspace too small
    assert lib.moe_preprocess(byref(routing), byref(good_shape), byref(good_layout), byref(handle), fake, 16,
                              None) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    # missing handle array
    h2 = moe._HandleDev(*([fake] * 7 + [None]))
    assert lib.moe_preprocess(byref(routing), byref(good_shape), byref(good_layout), byref(h2), fake, 1 << 30,
                              None) == moe.MOE_ERR_INVALID_ARG
    # H not a multiple of 128; misaligned rows; unknown dtype
    assert lib.moe_dispatch_permute(byref(handle), byref(moe._Shape(64, 100, 8, 2, 0)), byref(good_layout),
                                    moe.DTYPE_BF16, fake, None, byref(routing), fake, None, None,
                                    None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_permute(byref(handle), byref(good_shape), byref(good_layout), moe.DTYPE_BF16,
                                    ctypes.c_void_p(0x1008), None, byref(routing), fake, None, None,
                                    None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_permute(byref(handle), byref(good_shape), byref(good_layout), 99, fake, None,
                                    byref(routing), fake, None, None, None) == moe.MOE_ERR_INVALID_ARG
    # FP8 dispatch without output scales
    assert lib.moe_dispatch_permute(byref(handle), byref(good_shape), byref(good_layout), moe.DTYPE_BF16_TO_FP8,
                                    fake, None, byref(routing), fake, None, None, None) == moe.MOE_ERR_INVALID_ARG
    # grouped MLP: I not a multiple of 128, workspace misaligned, NVFP4 without globals
    assert lib.moe_grouped_mlp(byref(handle), byref(moe._Shape(64, 256, 8, 2, 100)), byref(good_layout),
                               moe.DTYPE_BF16, fake, None, fake, None, fake, None, None, fake, 1 << 30, fake,
                               None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_grouped_mlp(byref(handle), byref(good_shape), byref(good_layout), moe.DTYPE_BF16, fake, None,
                               fake, None, fake, None, None, ctypes.c_void_p(0x1010), 1 << 30, fake,
                               None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_grouped_mlp(byref(handle), byref(good_shape), byref(good_layout), moe.DTYPE_NVFP4, fake, fake,
                               fake, fake, fake, fake, None, fake, 1 << 30, fake, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_grouped_mlp(byref(handle), byref(good_shape), byref(good_layout), moe.DTYPE_BF16, fake, None,
                               fake, None, fake, None, None, fake, 8, fake,
                               None) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    # NVFP4 stages 256 K elements: I = 128 (valid for bf16 and FP8) is not built for it
    glob = moe._Nvfp4Globals(fake, fake, fake, fake)
    assert lib.moe_grouped_mlp(byref(handle), byref(good_shape), byref(good_layout), moe.DTYPE_NVFP4, fake, fake,
                               fake, fake, fake, fake, byref(glob), fake, 1 << 30, fake,
                               None) == moe.MOE_ERR_UNSUPPORTED
    assert lib.moe_grouped_mlp(byref(handle), byref(moe._Shape(64, 384, 8, 2, 256)), byref(good_layout),
                               moe.DTYPE_NVFP4, fake, fake, fake, fake, fake, fake, byref(glob), fake, 1 << 30,
                               fake, None) == moe.MOE_ERR_UNSUPPORTED
    # extended grouped MLP: misaligned FC2 row probabilities, unknown output format, MX output without scales
    assert lib.moe_grouped_mlp_ex(byref(handle), byref(good_shape), byref(good_layout), moe.DTYPE_BF16, fake, None,
                                  fake, None, fake, None, None, fake, 1 << 30, moe.COMBINE_BF16, fake, None,
                                  ctypes.c_void_p(0x1002), None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_grouped_mlp_ex(byref(handle), byref(good_shape), byref(good_layout), moe.DTYPE_BF16, fake, None,
                                  fake, None, fake, None, None, fake, 1 << 30, 9, fake, None, fake,
                                  None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_grouped_mlp_ex(byref(handle), byref(good_shape), byref(good_layout), moe.DTYPE_FP8_E4M3_B128,
                                  fake, fake, fake, fake, fake, fake, None, fake, 1 << 30, moe.COMBINE_MXFP8, fake,
                                  None, fake, None) == moe.MOE_ERR_INVALID_ARG
    # backward calls: null gradient buffers, probability gradients without their inputs, unknown routing format
    assert lib.moe_combine_backward(byref(handle), byref(good_shape), byref(good_layout), fake, fake, fake, None,
                                    None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_combine_backward(byref(handle), byref(good_shape), byref(good_layout), fake, None, fake, fake,
                                    fake, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_combine_backward(byref(handle), byref(good_shape), byref(good_layout), fake, fake, None, fake,
                                    fake, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_backward(byref(handle), byref(good_shape), byref(good_layout), 5, fake, None, fake,
                                     None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_backward(byref(handle), byref(good_shape), byref(good_layout), 0, fake, fake, fake,
                                     None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_backward(byref(handle), byref(good_shape), byref(good_layout), 0, None, None, fake,
                                     None, None) == moe.MOE_ERR_INVALID_ARG
    # combine with a null expert buffer
    assert lib.moe_combine_unpermute(byref(handle), byref(good_shape), byref(good_layout), None, None, fake,
                                     None) == moe.MOE_ERR_INVALID_ARG
    # quantizers: shapes not multiples of the block
    assert lib.moe_quantize_fp8_blocks(fake, 1, 100, 128, fake, fake, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_nvfp4_rows(fake, 4, 24, fake, fake, fake, None) == moe.MOE_ERR_INVALID_ARG


def test_ring_rotation_and_lifetime_errors(moe):
    """Round-robin slots; acquiring a held slot is early reuse; releasing a
    free slot is a double release; neither changes the ring."""
    r = moe.Ring(3, use_events=False)
    assert [r.acquire(), r.acquire(), r.acquire()] == [0, 1, 2]
    with pytest.raises(moe.MoeError) as ei:
        r.acquire()
    assert ei.value.status == moe.MOE_ERR_RING_EARLY_REUSE
    r.release(0)
    with pytest.raises(moe.MoeError) as ei:
        r.release(0)
    assert ei.value.status == moe.MOE_ERR_RING_DOUBLE_RELEASE
    assert r.acquire() == 0          # slot 0 is free again, next in order
    with pytest.raises(moe.MoeError) as ei:
        r.acquire()                  # slot 1 is still held by its first producer
    assert ei.value.status == moe.MOE_ERR_RING_EARLY_REUSE
    r.release(1)
    r.release(2)
    assert r.acquire() == 1
    with pytest.raises(moe.MoeError):
        r.release(7)
    r.close()
    with pytest.raises(moe.MoeError):
        moe.Ring(0, use_events=False)


def test_debug_hook_arguments(moe):
    """The fused-MLP testing hook takes a token tile or -1 (cancel); anything
    below -1 is rejected on the host."""
    moe.moe_debug_next_grouped_mlp_silent_token_tile(-1)
    with pytest.raises(moe.MoeError):
        moe.moe_debug_next_grouped_mlp_silent_token_tile(-2)


def test_decode_bucket_selection(moe):
    """Smallest bucket that holds the batch; zero tokens keep the smallest
    bucket (a non-empty launch); above the largest bucket, or a malformed
    ladder, is an argument error."""
    ladder = [1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096, 8192]
    assert moe.moe_decode_bucket(0, ladder) == 1
    assert moe.moe_decode_bucket(1, ladder) == 1
    assert moe.moe_decode_bucket(37, ladder) == 64
    assert moe.moe_decode_bucket(64, ladder) == 64
    assert moe.moe_decode_bucket(65, ladder) == 128
    assert moe.moe_decode_bucket(8192, ladder) == 8192
    assert moe.moe_decode_bucket(100, [64, 256, 8192]) == 256
    for bad in ((8193, ladder), (-1, ladder), (5, []), (5, [4, 4, 8]), (5, [8, 4]), (5, [0, 4])):
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_decode_bucket(*bad)
        assert ei.value.status == moe.MOE_ERR_INVALID_ARG
