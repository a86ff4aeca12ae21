"""Host-side pieces of bench.py that need no GPU: the validity key of the
committed ncu capture (roofline traffic) follows code edits, not comment
edits."""
import importlib.util
import os
import shutil

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_host_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _copy_sources(dst):
    src_csrc = os.path.join(ROOT, "microscaling_quantized_convolution_only_b300", "csrc")
    shutil.copytree(src_csrc, os.path.join(dst, "microscaling_quantized_convolution_only_b300", "csrc"))
    os.makedirs(os.path.join(dst, "include"))
    shutil.copy(os.path.join(ROOT, "include", "mqconv.h"), os.path.join(dst, "include", "mqconv.h"))
    return os.path.join(dst, "microscaling_quantized_convolution_only_b300", "csrc", "conv_halo.cuh")


def test_sources_key_ignores_comments_not_code(tmp_path):
    b = _bench()
    ref = b.kernel_sources_sha1()
    f = _copy_sources(str(tmp_path))
    assert b.kernel_sources_sha1(str(tmp_path)) == ref
    text = open(f).read()
    open(f, "w").write("// an added comment line\n/* and a block\n comment */\n" + text.replace("\n", "\n\n", 3))
    assert b.kernel_sources_sha1(str(tmp_path)) == ref
    open(f, "w").write(text.replace("constexpr int DSTAGES = 2;", "constexpr int DSTAGES = 3;"))
    assert b.kernel_sources_sha1(str(tmp_path)) != ref


def test_traffic_scales_with_batch_and_needs_matching_sources():
    b = _bench()
    key = ("stack4-56x56-c128-nvfp4", "conv_dgrad")
    t = b.TRAFFIC[key]
    if t["sources_sha1"] == b.kernel_sources_sha1(names=b.CONV_SOURCES):
        assert b.captured_traffic(*key, t["batch"] * 4) == t["bytes_per_launch"] * 4
    else:
        assert b.captured_traffic(*key, t["batch"]) is None
    assert b.captured_traffic("no-such-workload", "conv_dgrad", 64) is None


def test_conv_key_covers_the_conv_sources_only(tmp_path):
    """The conv traffic key follows the conv kernels' sources: an edit to
    the quantizer leaves it, an edit to a conv source changes it."""
    b = _bench()
    ref = b.kernel_sources_sha1(names=b.CONV_SOURCES)
    f = _copy_sources(str(tmp_path))
    csrc = os.path.dirname(f)
    q = os.path.join(csrc, "quantize.cu")
    open(q, "w").write(open(q).read().replace("constexpr int QT_STAGES = 2;", "constexpr int QT_STAGES = 3;"))
    assert b.kernel_sources_sha1(str(tmp_path), names=b.CONV_SOURCES) == ref
    assert b.kernel_sources_sha1(str(tmp_path)) != b.kernel_sources_sha1()
    open(f, "w").write(open(f).read().replace("constexpr int DSTAGES = 2;", "constexpr int DSTAGES = 3;"))
    assert b.kernel_sources_sha1(str(tmp_path), names=b.CONV_SOURCES) != ref
