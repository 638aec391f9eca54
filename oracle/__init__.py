"""CPU oracle for the paged GQA decode and page-budgeting path (test infrastructure only)."""
