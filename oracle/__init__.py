"""CPU oracle for the NVFP4 block-scaled path.  Test infrastructure only: the
library never imports it.  See nvfp4_oracle.py."""
from . import nvfp4_oracle  # noqa: F401
