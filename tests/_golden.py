"""Reader for the small text fixtures under tests/golden/ ("key: value" lines)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, value = line.partition(":")
            parts = value.split()
            nums = [float(p) for p in parts]
            out[key.strip()] = nums[0] if len(nums) == 1 else nums
    return out
