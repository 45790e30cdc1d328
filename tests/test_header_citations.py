"""Every method call of the C ABI states the passage of the source pages it
follows: the comment block that documents a declaration in include/zero.h
must carry a section citation ("§").  Exempt are the calls that are not part
of the method: handle release, status strings, the error message, the
profiling and device-byte counters, the test hook, and the allocation-free
entry point (which has no counterpart on the pages)."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "zero.h")

EXEMPT = {"zero_flat_free", "zero_group_free", "zero_status_string", "zero_last_error",
          "zero_flat_profile_enable", "zero_flat_profile_read", "zero_flat_profile_reduce_form",
          "zero_flat_device_bytes",
          "zero_shard_step_noalloc"}

DECL = re.compile(r"^(?:const\s+)?(?:zero_status|uint64_t|const char)\s*\*?\s*(zero_\w+)\s*\(",
                  re.M)


def documented_declarations(text):
    """(name, the comment block in front of it) for every declaration; a
    comment block documents every declaration that follows it up to the next
    comment block."""
    out = []
    for mt in DECL.finditer(text):
        head = text[:mt.start()]
        end = head.rfind("*/")
        start = head.rfind("/*", 0, end) if end >= 0 else -1
        out.append((mt.group(1), head[start:end + 2] if start >= 0 else ""))
    return out


def test_parser_sees_the_boundary():
    names = [n for n, _ in documented_declarations(open(HEADER).read())]
    for want in ("zero_flat_init", "zero_flat_layout", "zero_shard_step", "zero_shard_reduce",
                 "zero_shard_apply", "zero_loss_scaler_state", "zero_set_loss_scaler_state",
                 "zero_memory_bytes", "zero_flat_free"):
        assert want in names


def test_parser_catches_a_missing_citation():
    text = ("/* cites §3.3 */\nzero_status zero_a(int x);\n"
            "/* no citation here */\nzero_status zero_b(int x);\n")
    got = dict(documented_declarations(text))
    assert "§" in got["zero_a"] and "§" not in got["zero_b"]


def test_every_method_call_cites_its_passage():
    missing = [n for n, block in documented_declarations(open(HEADER).read())
               if n not in EXEMPT and "§" not in block]
    assert not missing, "declarations without a passage citation: %s" % missing
